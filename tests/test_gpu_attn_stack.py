"""GPU tests of the stack with the causal attention core in place of the
repeat(v) stand-in (ws_stack_cfg.attn = WS_ATTN_CAUSAL).

- One step of a 2-layer stack with the 0.5B widths matches the fp64 oracle's
  stack in the same mode: loss, every adapter gradient (q and k now carry
  gradient) and the Adam update.
- Inside that step the attention forward and backward match the oracle fed
  the GPU's own saved q, k, v and the o projection's bf16 input gradient dO
  (the layer the backward processed last, layer 0).
- Streamed (2-slot window, recompute) equals resident bitwise over 3 steps
  on loss, gradients, parameters and both Adam moments (research page
  "Poros", result paragraph: the comparison is torch.equal).
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_to_dev, dev, f32_to_dev, rel, to_f64

pytestmark = pytest.mark.gpu

STACK_TOL = 1e-2
NAMES = ("q", "k", "v", "o", "gate", "up", "down")


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _fns(seed):
    from weight_streaming_nf4_gb300 import synth

    def wfn(layer, lin, N, K):
        W, _, _ = synth.stack_weights(seed, layer, NAMES[lin], N, K)
        return bf16_to_dev(W)

    def pfn(layer, lin, N, K):
        _, A, B = synth.stack_weights(seed, layer, NAMES[lin], N, K)
        return f32_to_dev(A), f32_to_dev(B)
    return wfn, pfn


def _h0(cfg, step):
    from weight_streaming_nf4_gb300 import synth
    return f32_to_dev(synth.stack_h0(cfg.seed, step, cfg.M, cfg.H))


def _oracle_params(orc, cfg, seed):
    from weight_streaming_nf4_gb300 import synth
    Wq, As, Bs = [], [], []
    for layer in range(cfg.n_layers):
        for lin, (N, K) in enumerate(cfg.shapes()):
            W, A, B = synth.stack_weights(seed, layer, NAMES[lin], N, K)
            Wq.append(orc.dequant_nf4(*orc.quantize_nf4(W)))
            As.append(A)
            Bs.append(B)
    return Wq, As, Bs


def test_attention_stack_step_matches_oracle(ops, orc):
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=192, H=896, KV=128, I=4864, head_dim=64, n_layers=2,
                       attn=ops.ATTN_CAUSAL)
    wfn, pfn = _fns(5)
    run = StackRun(cfg, 2, False, wfn, pfn)
    p0 = run.params.clone()
    step, lr = 4, 2e-4
    run.step(step, _h0(cfg, step), lr=lr)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    Wq, As, Bs = _oracle_params(orc, cfg, 5)
    ocfg = orc.StackCfg(M=cfg.M, H=cfg.H, KV=cfg.KV, I=cfg.I, head_dim=cfg.head_dim,
                        n_layers=cfg.n_layers, p=cfg.p, attn=1)
    h0 = synth.stack_h0(cfg.seed, step, cfg.M, cfg.H).astype(np.float64)
    loss, _, dA, dB = orc.stack_fwd_bwd(ocfg, step, Wq, As, Bs, h0)
    assert abs(float(run.loss.item()) - loss) <= 1e-4 * abs(loss)
    for layer in range(cfg.n_layers):
        for lin in range(7):
            gA = to_f64(run.param(layer, lin, "A", run.grads))
            gB = to_f64(run.param(layer, lin, "B", run.grads))
            i = layer * 7 + lin
            assert np.any(gB != 0), (layer, NAMES[lin])
            assert rel(gA, dA[i]) <= STACK_TOL, (layer, NAMES[lin], "A", rel(gA, dA[i]))
            assert rel(gB, dB[i]) <= STACK_TOL, (layer, NAMES[lin], "B", rel(gB, dB[i]))
    p = to_f64(p0)
    g = to_f64(run.grads)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    orc.adam_step(p, g, m, v, step + 1, lr=lr)
    got = to_f64(run.params)
    assert rel(got - to_f64(p0), p - to_f64(p0)) <= 1e-5

    # the attention of layer 0 on the GPU's own saved inputs
    M, H, KV, hd = cfg.M, cfg.H, cfg.KV, cfg.head_dim
    sv = run.saved.cpu().numpy()

    def field(name, shape, dtype, layer=0):
        off = layer * run.sizes["saved_layer"] + ops.stack_saved_offset(cfg, name)
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return sv[off:off + n].view(dtype).reshape(shape)

    def bf(b):
        return synth.bf16_bits_to_f32(b).astype(np.float64)

    q, k, v = bf(field("q", (M, H), np.uint16)), bf(field("k", (M, KV), np.uint16)), \
        bf(field("v", (M, KV), np.uint16))
    o_ref, lse_ref = orc.attention_fwd(q, k, v, 1, hd, want_lse=True)
    assert rel(field("o32", (M, H), np.float32).astype(np.float64), o_ref) <= 1e-4
    np.testing.assert_array_equal(field("vr", (M, H), np.uint16),
                                  synth.to_bf16_bits(field("o32", (M, H), np.float32)))
    np.testing.assert_allclose(field("lse", (H // hd, M), np.float32), lse_ref, rtol=1e-5,
                               atol=1e-5)
    ws = run.workspace.cpu().numpy()

    def wk(name, shape):
        off = ops.stack_workspace_offset(cfg, 2, name)
        return bf(ws[off:off + int(np.prod(shape)) * 2].view(np.uint16).reshape(shape))

    dq_ref, dk_ref, dv_ref = orc.attention_bwd(q, k, v, wk("do", (M, H)), 1, hd)
    assert rel(wk("dq", (M, H)), dq_ref) <= TOL
    assert rel(wk("dk", (M, KV)), dk_ref) <= TOL
    assert rel(wk("dv", (M, KV)), dv_ref) <= TOL


def test_attention_stack_streamed_equals_resident(ops):
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=512, H=896, KV=128, I=4864, head_dim=64, n_layers=8,
                       attn=ops.ATTN_CAUSAL)
    wfn, pfn = _fns(6)
    res = StackRun(cfg, 2, False, wfn, pfn)
    stm = StackRun(cfg, 2, True, wfn, pfn)
    for step in range(3):
        h0 = _h0(cfg, step)
        res.step(step, h0)
        stm.step(step, h0)
        torch.cuda.synchronize()
        assert torch.equal(res.loss, stm.loss), step
        assert torch.equal(res.grads, stm.grads), step
    assert ops.device_error() == 0
    for name in ("params", "grads", "adam_m", "adam_v"):
        assert torch.equal(getattr(res, name), getattr(stm, name)), name
    assert np.isfinite(float(res.loss.item()))


@pytest.mark.parametrize("order", ["mb", "block"])
def test_attention_stack_grad_accumulation_bitwise(ops, order):
    """Gradient accumulation over 2 micro-batches with the attention core:
    streamed (either order) equals resident bitwise over 2 steps."""
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=256, H=896, KV=128, I=4864, head_dim=64, n_layers=4,
                       attn=ops.ATTN_CAUSAL)
    o = ops.GA_MICROBATCH_MAJOR if order == "mb" else ops.GA_BLOCK_MAJOR
    wfn, pfn = _fns(7)
    res = StackRun(cfg, 2, False, wfn, pfn, n_micro=2, order=o)
    stm = StackRun(cfg, 2, True, wfn, pfn, n_micro=2, order=o)
    from weight_streaming_nf4_gb300 import synth
    for step in range(2):
        h0 = torch.cat([f32_to_dev(synth.stack_h0(cfg.seed + mb, step, cfg.M, cfg.H)).reshape(-1)
                        for mb in range(2)])
        res.step(step, h0)
        stm.step(step, h0)
        torch.cuda.synchronize()
        assert torch.equal(res.loss, stm.loss), step
        assert torch.equal(res.grads, stm.grads), step
    assert ops.device_error() == 0
    for name in ("params", "adam_m", "adam_v"):
        assert torch.equal(getattr(res, name), getattr(stm, name)), name
