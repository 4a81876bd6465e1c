"""The tensor-pipe probe behind the roofline's own BF16 peak (include/gdn.h,
gdn_tensor_probe): its FLOP count, its error word and argument checks, and a
measured rate inside the physical range of one GB300."""
import pytest

import torch

import linear_attention_gdn_gb300 as gdn

pytestmark = pytest.mark.gpu


def test_tensor_probe_counts_and_rate():
    dev = torch.device("cuda", 0)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gdn.gdn_tensor_probe(100, err)   # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    flops = gdn.gdn_tensor_probe(4000, err)
    e1.record()
    e1.synchronize()
    assert int(err.item()) == 0
    assert flops == 2.0 * 128 * 256 * 16 * 4 * 4000 * sms
    tflops = flops / e0.elapsed_time(e1) / 1e9
    # dense BF16 on one GB300: a few hundred TFLOP/s at the very least, and no more than the
    # 152 SMs x 8,192 FLOP per cycle at 2.1 GHz that the tensor cores can issue
    assert 200.0 < tflops < 2700.0, tflops


@pytest.mark.parametrize("iters", [0, -1, (1 << 20) + 1])
def test_tensor_probe_rejects_bad_iteration_counts(iters):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gdn.GDNError):
        gdn.gdn_tensor_probe(iters, err)
