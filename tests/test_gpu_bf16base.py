"""The bf16-base mode (the pages' bf16 streaming, "Limitations", section
"bf16 LoRA (EXPERIMENTAL)": same engine and GEMM, the frozen weights stream
as bf16, 2 bytes per weight, and the streamed run is still bitwise equal to
the resident one).  The dequant GEMM's producer is replaced by TMA loads of
the bf16 weight tiles; parity is the NF4 path's minus the codec: the oracle
is fed the bf16 weight itself.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_to_dev, f32_to_dev, rel, to_f64
from test_gpu_stack import STACK_TOL, _fns

pytestmark = pytest.mark.gpu
P = 0.1


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


@pytest.mark.parametrize("M,N,K", [(64, 512, 512), (300, 896, 1088), (512, 128, 896),
                                   (512, 5120, 5120), (640, 2048, 1024), (200, 4864, 896)])
def test_bf16_linear_fwd_bwd_parity(ops, orc, M, N, K):
    from weight_streaming_nf4_gb300 import synth
    d = synth.linear_inputs(3, M, N, K, 16, tag=f"bf{M}x{N}x{K}")
    W = ops.Bf16Weight(bf16_to_dev(d["W"]), N, K)
    key = ops.dropout_key(seed=3, step=2, layer=1, linear=4, p=P)
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])
    y, U, mask = ops.lora_linear_fwd(W, x, A, B, key)
    dX, dA, dB = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY)
    dXf, _, _ = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX_f32=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    om = orc.dropout_mask(3, 2, 1, 4, 0, P, M, K)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), om)
    s = 2.0 / (1.0 - P)
    yo, Uo = orc.lora_fwd(d["x"], d["W"], d["A"], d["B"], om, s)
    dXo, dAo, dBo = orc.lora_bwd(d["x"], d["W"], d["A"], d["B"], om, d["dY"], s)
    assert rel(to_f64(y), yo) <= TOL
    assert rel(to_f64(U), Uo) <= 1e-5
    assert rel(to_f64(dX), dXo) <= TOL
    assert rel(to_f64(dXf), dXo) <= 1e-4
    assert rel(to_f64(dA), dAo) <= TOL and rel(to_f64(dB), dBo) <= TOL


def test_bf16_weight_through_gemm_is_exact(ops):
    """x = unit rows e_k, B = 0: y[m, :] = W[:, k_m] bit for bit (the weight
    tile reaches the tensor cores unchanged)."""
    from weight_streaming_nf4_gb300 import synth
    M, N, K = 512, 768, 1024
    Wb = synth.normal_bf16(5, "bfpin", (N, K), 0.02)
    rng = np.random.default_rng(1)
    ks = rng.integers(0, K, size=M)
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), ks] = synth.to_bf16_bits(np.array([1.0]))[0]
    W = ops.Bf16Weight(bf16_to_dev(Wb), N, K)
    y, _, _ = ops.lora_linear_fwd(W, bf16_to_dev(x), f32_to_dev(np.zeros((16, K), np.float32)),
                                  f32_to_dev(np.zeros((N, 16), np.float32)), ops.dropout_key(p=0.0))
    got = y.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, Wb[:, ks].T)


def _bf16_fns(seed):
    wfn, pfn = _fns(seed)
    return wfn, pfn


def test_bf16_streamed_equals_resident_bitwise(ops):
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=512, H=896, KV=128, I=4864, head_dim=64, n_layers=8, base=ops.BASE_BF16)
    wfn, pfn = _bf16_fns(8)
    stm = StackRun(cfg, 2, True, wfn, pfn)
    res = StackRun(cfg, 2, False, wfn, pfn, image_from=stm)
    from test_gpu_stack import _h0
    for step in range(10):
        h0 = _h0(cfg, step)
        res.step(step, h0)
        stm.step(step, h0)
        torch.cuda.synchronize()
        assert torch.equal(res.loss, stm.loss), step
        assert torch.equal(res.grads, stm.grads), step
    for name in ("params", "adam_m", "adam_v"):
        assert torch.equal(getattr(res, name), getattr(stm, name)), name
    assert ops.device_error() == 0


def test_bf16_step_matches_oracle(ops, orc):
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=128, H=896, KV=128, I=4864, head_dim=64, n_layers=2, base=ops.BASE_BF16)
    wfn, pfn = _bf16_fns(9)
    run = StackRun(cfg, 2, False, wfn, pfn)
    step = 3
    from test_gpu_stack import _h0
    run.step(step, _h0(cfg, step), lr=0.0)
    torch.cuda.synchronize()
    names = ("q", "k", "v", "o", "gate", "up", "down")
    Wq, As, Bs = [], [], []
    for layer in range(cfg.n_layers):
        for lin, (N, K) in enumerate(cfg.shapes()):
            W, A, B = synth.stack_weights(9, layer, names[lin], N, K)
            Wq.append(W)   # bf16 base: the weight itself
            As.append(A)
            Bs.append(B)
    ocfg = orc.StackCfg(M=cfg.M, H=cfg.H, KV=cfg.KV, I=cfg.I, head_dim=cfg.head_dim,
                        n_layers=cfg.n_layers, p=cfg.p)
    h0 = synth.stack_h0(cfg.seed, step, cfg.M, cfg.H).astype(np.float64)
    loss, _, dA, dB = orc.stack_fwd_bwd(ocfg, step, Wq, As, Bs, h0)
    assert abs(float(run.loss.item()) - loss) <= 1e-4 * abs(loss)
    for layer in range(cfg.n_layers):
        for lin in range(2, 7):
            i = layer * 7 + lin
            assert rel(to_f64(run.param(layer, lin, "A", run.grads)), dA[i]) <= STACK_TOL
            assert rel(to_f64(run.param(layer, lin, "B", run.grads)), dB[i]) <= STACK_TOL


def test_bf16_loader_copies_weights(ops):
    """ws_stack_put_weight with a bf16 base copies the weight into place as it is."""
    from weight_streaming_nf4_gb300 import synth
    cfg = ops.StackCfg(M=64, H=256, KV=64, I=512, head_dim=32, n_layers=2, base=ops.BASE_BF16)
    bb = ops.stack_sizes(cfg, 1)["block_bytes"]
    host = torch.zeros(2 * bb, dtype=torch.uint8, pin_memory=True)
    W = synth.normal_bf16(1, "bfload", (512, 256), 0.02)
    ops.stack_put_weight(cfg, 1, 1, 5, bf16_to_dev(W), host)
    torch.cuda.synchronize()
    oc, oa = ops.stack_weight_offset(cfg, 0, 5)
    assert oc == oa
    got = host[bb + oc:bb + oc + W.size * 2].numpy().view(np.uint16).reshape(W.shape)
    assert np.array_equal(got, W)
