"""Failure detection on the GPU without a fault.

Every wait inside the library's kernels is bounded: when it runs out the
kernel records a bit in the device error word, lets its copies land, frees
its tensor memory and returns, so the CUDA context stays usable and the
host learns of it through ws_device_error.  The self-check entry point runs
the stream-K finisher's bounded wait on a word that nothing sets, with a
one-millisecond limit; nothing traps or faults.
"""
import pytest
import torch

from gpu_util import TOL, bf16_to_dev, f32_to_dev, rel, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def test_bounded_wait_gives_up_and_the_context_stays_usable(ops, orc):
    from weight_streaming_nf4_gb300 import synth
    assert ops.device_error() == 0
    ops.selfcheck_bounded_wait(1000)
    flags = ops.device_error()                 # synchronises, reads and clears
    assert flags == ops.WS_DERR_TIMEOUT_PEER
    assert ops.device_error() == 0             # cleared
    # the next call runs normally and passes parity
    M, N, K, p = 128, 512, 1024, 0.1
    d = synth.linear_inputs(3, M, N, K, 16, tag="after_timeout")
    codes, absmax = ops.quantize_nf4(bf16_to_dev(d["W"]))
    W = ops.NF4Weight(codes, absmax, N, K)
    key = ops.dropout_key(seed=3, p=p)
    y, U, mask = ops.lora_linear_fwd(W, bf16_to_dev(d["x"]), f32_to_dev(d["A"]),
                                     f32_to_dev(d["B"]), key)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    Wq = orc.dequant_nf4(*orc.quantize_nf4(d["W"]))
    om = orc.dropout_mask(3, 0, 0, 0, 0, p, M, K)
    yo, _ = orc.lora_fwd(d["x"], Wq, d["A"], d["B"], om, 2.0 / (1.0 - p))
    assert rel(to_f64(y), yo) <= TOL


def test_work_after_an_unread_error_is_skipped_not_corrupted(ops):
    """Kernels that start while the error word is set skip their work (they
    leave outputs untouched) until the host reads and clears the word."""
    N, K, M = 256, 512, 64
    W = (torch.randn(N, K, device="cuda:0") * 0.02).to(torch.bfloat16)
    codes, absmax = ops.quantize_nf4(W)
    Wn = ops.NF4Weight(codes, absmax, N, K)
    act = torch.randn(M, K, device="cuda:0").to(torch.bfloat16)
    ops.selfcheck_bounded_wait(500)
    torch.cuda.synchronize()                   # the word is set before the next launch
    out = torch.full((M, N), 7.0, device="cuda:0", dtype=torch.float32)
    ops.nf4_matmul(Wn, act, out=out, out_f32=True)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())            # skipped
    assert ops.device_error() == ops.WS_DERR_TIMEOUT_PEER
    ops.nf4_matmul(Wn, act, out=out, out_f32=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert not bool((out == 7.0).any())
    with pytest.raises(ops.WsError) as e:
        ops.selfcheck_bounded_wait(0)
    assert e.value.status == -1
