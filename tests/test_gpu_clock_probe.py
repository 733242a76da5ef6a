"""attn_sm_clock_sample, the timing helper the benchmark reads SM clocks with: nearly
every SM records a sample, and two samples around some work give an average SM clock
within the part's range."""
import pytest
import torch

import sage_attention_forward_gb300 as sa

pytestmark = pytest.mark.gpu


def test_sm_clock_sample(cuda_dev):
    n_sms = torch.cuda.get_device_properties(cuda_dev).multi_processor_count
    n = n_sms + 32
    a = sa.sm_clock_sample(torch.empty((n, 2), dtype=torch.int64, device=cuda_dev))
    x = torch.randn(4096, 4096, device=cuda_dev)
    for _ in range(20):
        x = (x @ x).clamp_(-1, 1)
    b = sa.sm_clock_sample(torch.empty((n, 2), dtype=torch.int64, device=cuda_dev))
    torch.cuda.synchronize()
    ha, hb = a.cpu().numpy(), b.cpu().numpy()
    assert (ha[:, 0] > 0).sum() >= 0.9 * n_sms and (hb[:, 0] > 0).sum() >= 0.9 * n_sms
    mhz = sa.sm_clock_mhz(ha, hb)
    assert mhz is not None and 300.0 < mhz < 2500.0, mhz
    with pytest.raises(ValueError):
        sa.sm_clock_sample(torch.empty((n, 3), dtype=torch.int64, device=cuda_dev))
