"""The library's calls inside a CUDA graph (CUDA through the C ABI): every entry
point only enqueues work on the caller's stream (tensor maps travel by value in
the kernel parameters, nothing is allocated or synchronised), so a
torch.cuda.CUDAGraph captures attn_fwd_bf16, the one-call Sage op in both P V
modes and the two-call path, and its replays reproduce eager calls bit for
bit, also after new values are written into the captured input buffers."""
import pytest
import torch

import sage_attention_forward_gb300 as sa
from workloads import make_inputs, small_case, to_device

pytestmark = pytest.mark.gpu


def run_all(q, k, v, outs, ws):
    sa.attn_fwd_bf16(q, k, v, out=outs["bf16"])
    sa.sage_attention(q, k, v, out=outs["sage"], workspace=ws["sage"])
    sa.sage_attention(q, k, v, out=outs["pv16"], workspace=ws["pv16"], pv="bf16")
    prep = sa.sage_prepare(q, k, v, out=ws["prep"], workspace=ws["prep_ws"])
    sa.sage_attn_fwd(prep, out=outs["two"], workspace=ws["attn_ws"])


@pytest.mark.parametrize("B,H,S", [(1, 2, 512), (2, 3, 1000)])
def test_graph_replay_matches_eager(cuda_dev, B, H, S):
    inp = make_inputs(small_case(B, H, S, 2000 + S))
    g = to_device(inp, cuda_dev)
    q, k, v = g.q.clone(), g.k.clone(), g.v.clone()
    S_pad = sa.sage_padded_len(S)
    outs = {n: torch.empty_like(q) for n in ("bf16", "sage", "pv16", "two")}
    ws = {"sage": sa.sage_attention_workspace(B, H, S, cuda_dev),
          "pv16": sa.sage_attention_workspace(B, H, S, cuda_dev, pv="bf16"),
          "prep": sa.Prepared.empty(B, H, S, S_pad, cuda_dev),
          "prep_ws": sa.prepare_workspace(B, H, cuda_dev, S_pad),
          "attn_ws": sa.attn_workspace(B, H, S_pad, cuda_dev)}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                 # warm-up outside the capture (first-use setup)
        run_all(q, k, v, outs, ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = {n: t.clone() for n, t in outs.items()}

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_all(q, k, v, outs, ws)
    for t in outs.values():
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    for n in outs:
        assert torch.equal(outs[n].view(torch.int16), eager[n].view(torch.int16)), n

    # new inputs in the captured buffers: the replay computes on them
    inp2 = to_device(make_inputs(small_case(B, H, S, 3000 + S)), cuda_dev)
    q.copy_(inp2.q)
    k.copy_(inp2.k)
    v.copy_(inp2.v)
    graph.replay()
    torch.cuda.synchronize()
    replayed = {n: t.clone() for n, t in outs.items()}
    run_all(q, k, v, outs, ws)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    for n in outs:
        assert torch.equal(replayed[n].view(torch.int16), outs[n].view(torch.int16)), n
        assert not torch.equal(replayed[n], eager[n]), n
