"""GPU tests of the block engine: block forward / backward with
recompute, the streamed training step, and the pinned-host block copy.

- The recompute (the forward run again from the block-boundary activation
  with the same Philox keys) reproduces the kept intermediates bit for bit,
  so the recomputed backward equals the resident backward exactly (research
  page "Poros", RNG-capture paragraph).
- A streamed run equals a resident run bitwise on loss, gradients,
  parameters and both Adam moments over 20 steps (research page "Poros",
  result paragraph: the comparison is torch.equal, not a tolerance).
- Every forward and every backward operation of a layer matches the oracle
  fed the GPU's own inputs (within TOL, or one bf16 ulp, or exactly).
- One step of a 2-layer stack matches the fp64 oracle within STACK_TOL.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_to_dev, dev, f32_to_dev, rel, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _fns(seed=0):
    from weight_streaming_nf4_gb300 import synth
    names = ("q", "k", "v", "o", "gate", "up", "down")

    def wfn(layer, lin, N, K):
        W, _, _ = synth.stack_weights(seed, layer, names[lin], N, K)
        return bf16_to_dev(W)

    def pfn(layer, lin, N, K):
        _, A, B = synth.stack_weights(seed, layer, names[lin], N, K)
        return f32_to_dev(A), f32_to_dev(B)
    return wfn, pfn


def _h0(cfg, step):
    from weight_streaming_nf4_gb300 import synth
    return f32_to_dev(synth.stack_h0(cfg.seed, step, cfg.M, cfg.H))


def test_recompute_backward_equals_saved_backward(ops):
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=200, H=256, KV=64, I=512, head_dim=32, n_layers=2)
    wfn, pfn = _fns(1)
    run = StackRun(cfg, 2, False, wfn, pfn)
    sz = run.sizes
    M, H = cfg.M, cfg.H
    h0 = _h0(cfg, 3)
    h1 = torch.empty(M * H, device=dev())
    saved = torch.empty(2 * sz["saved_layer"], dtype=torch.uint8, device=dev())
    ops.block_forward(cfg, run.dev_weights, 0, 2, run.params, 3, h0, h1, saved, run.workspace)
    h1b = torch.empty_like(h1)
    ops.block_forward(cfg, run.dev_weights, 0, 2, run.params, 3, h0, h1b, None, run.workspace)
    assert torch.equal(h1, h1b)
    dh = torch.randn(M * H, device=dev()) * 1e-3
    g1 = torch.zeros_like(run.params)
    g2 = torch.zeros_like(run.params)
    dh1 = torch.empty_like(dh)
    dh2 = torch.empty_like(dh)
    ops.block_backward_recompute(cfg, run.dev_weights, 0, 2, run.params, 3, h0, saved, dh, dh1, g1,
                                 run.workspace)
    ops.block_backward_recompute(cfg, run.dev_weights, 0, 2, run.params, 3, h0, None, dh, dh2, g2,
                                 run.workspace)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert torch.equal(dh1, dh2)
    assert torch.equal(g1, g2)
    assert float(g1.abs().sum()) > 0


# End-to-end tolerance of a whole step against the oracle.  Both sides round
# to bf16 at the same storage points (a, v, o, b, gate, up, act, down per
# layer forward; dY of down, gate, up, o, v per layer backward), but their
# pre-rounding values differ by fp32-versus-fp64 accumulation, and once a
# value lands on the other side of a rounding boundary the difference is one
# bf16 ulp (2^-8 relative) that later layers carry on.  Each storage point
# can therefore add up to the bf16 rounding noise itself (about 1.5e-3
# normwise); over the ~20 points between the loss and the first layer's
# adapters these add in quadrature to about sqrt(20) * 1.5e-3 = 6.7e-3.
# Single operations are held to TOL, one bf16 ulp or exactly on their own
# (test_forward_local_parity, test_backward_local_parity).
STACK_TOL = 1e-2


def _oracle_params(orc, cfg, seed):
    from weight_streaming_nf4_gb300 import synth
    names = ("q", "k", "v", "o", "gate", "up", "down")
    Wq, As, Bs = [], [], []
    for layer in range(cfg.n_layers):
        for lin, (N, K) in enumerate(cfg.shapes()):
            W, A, B = synth.stack_weights(seed, layer, names[lin], N, K)
            Wq.append(orc.dequant_nf4(*orc.quantize_nf4(W)))
            As.append(A)
            Bs.append(B)
    return Wq, As, Bs


def test_one_step_matches_oracle(ops, orc):
    """Loss, every adapter gradient and the Adam update of one step of a
    2-layer stack with the 0.5B widths (H 896, kv 128, I 4864, head_dim 64)."""
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=128, H=896, KV=128, I=4864, head_dim=64, n_layers=2)
    wfn, pfn = _fns(2)
    run = StackRun(cfg, 2, False, wfn, pfn)
    p0 = run.params.clone()
    step, lr = 5, 2e-4
    run.step(step, _h0(cfg, step), lr=lr)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    Wq, As, Bs = _oracle_params(orc, cfg, 2)
    ocfg = orc.StackCfg(M=cfg.M, H=cfg.H, KV=cfg.KV, I=cfg.I, head_dim=cfg.head_dim,
                        n_layers=cfg.n_layers, p=cfg.p)
    h0 = synth.stack_h0(cfg.seed, step, cfg.M, cfg.H).astype(np.float64)
    loss, _, dA, dB = orc.stack_fwd_bwd(ocfg, step, Wq, As, Bs, h0)
    assert abs(float(run.loss.item()) - loss) <= 1e-4 * abs(loss)
    names = ("q", "k", "v", "o", "gate", "up", "down")
    for layer in range(cfg.n_layers):
        for lin in range(7):
            gA = to_f64(run.param(layer, lin, "A", run.grads))
            gB = to_f64(run.param(layer, lin, "B", run.grads))
            i = layer * 7 + lin
            if lin in (0, 1):
                assert np.all(gA == 0) and np.all(gB == 0)
                continue
            assert rel(gA, dA[i]) <= STACK_TOL, (layer, names[lin], "A", rel(gA, dA[i]))
            assert rel(gB, dB[i]) <= STACK_TOL, (layer, names[lin], "B", rel(gB, dB[i]))
    # the Adam update from the GPU's own gradients, against the oracle's Adam
    p = to_f64(p0)
    g = to_f64(run.grads)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    orc.adam_step(p, g, m, v, step + 1, lr=lr)
    got = to_f64(run.params)
    assert rel(got - to_f64(p0), p - to_f64(p0)) <= 1e-5
    assert np.array_equal(got == to_f64(p0), p == to_f64(p0))  # q, k untouched


def test_forward_local_parity(ops, orc):
    """Each forward operation of each layer against the oracle, fed the
    GPU's own inputs from the saved activations: RMSNorm and SiLU*up to one
    bf16 ulp, repeat_kv exactly, every NF4-LoRA linear within TOL, masks and
    U bit-exact / within 1e-5."""
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=256, H=896, KV=128, I=4864, head_dim=64, n_layers=2)
    wfn, pfn = _fns(4)
    run = StackRun(cfg, 2, False, wfn, pfn)
    step = 9
    run.step(step, _h0(cfg, step), lr=0.0)
    torch.cuda.synchronize()
    Wq, As, Bs = _oracle_params(orc, cfg, 4)
    M, H, KV, I = cfg.M, cfg.H, cfg.KV, cfg.I
    slot = run.sizes["saved_layer"]
    sv = run.saved.cpu().numpy()
    s = 2.0 / (1.0 - cfg.p)

    def field(layer, name, shape, dtype, lin=0):
        off = layer * slot + ops.stack_saved_offset(cfg, name, lin)
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return sv[off:off + n].view(dtype).reshape(shape)

    def f(b):
        return synth.bf16_bits_to_f32(b).astype(np.float64)

    def ulp_close(a, b):
        d = np.abs(f(a) - f(b))
        return np.all(d <= np.abs(f(b)) * 2.0 ** -7 + 1e-30) and np.mean(a == b) > 0.99

    bnd = to_f64(run.boundary).reshape(-1, M, H)
    for layer in range(cfg.n_layers):
        base = layer * 7
        h = field(layer, "h", (M, H), np.float32).astype(np.float64)
        a = field(layer, "a", (M, H), np.uint16)
        a_ref, r1 = orc.rmsnorm_bf16(h, cfg.eps)
        assert ulp_close(a, a_ref)
        assert rel(field(layer, "rstd1", (M,), np.float32), r1) <= 1e-5
        for lin, (N, K) in enumerate(cfg.shapes()):
            mk = field(layer, "mask", (M, K // 32), np.uint32, lin)
            assert np.array_equal(mk, orc.dropout_mask(cfg.seed, step, layer, lin, 0, cfg.p, M, K))
        v = field(layer, "v", (M, KV), np.uint16)
        vo, Uv = orc.lora_fwd(a, Wq[base + 2], As[base + 2], Bs[base + 2],
                              field(layer, "mask", (M, H // 32), np.uint32, 2), s)
        assert rel(f(v), vo) <= TOL
        assert rel(field(layer, "lora_u", (M, 16), np.float32, 2), Uv) <= 1e-5
        vr = field(layer, "vr", (M, H), np.uint16)
        assert np.array_equal(vr, orc.repeat_kv(v, H, cfg.head_dim))
        h1 = field(layer, "h1", (M, H), np.float32).astype(np.float64)
        oo, _ = orc.lora_fwd(vr, Wq[base + 3], As[base + 3], Bs[base + 3],
                             field(layer, "mask", (M, H // 32), np.uint32, 3), s)
        assert rel(h1 - h, oo) <= TOL
        b = field(layer, "b", (M, H), np.uint16)
        b_ref, _ = orc.rmsnorm_bf16(h1, cfg.eps)
        assert ulp_close(b, b_ref)
        g = field(layer, "gate", (M, I), np.uint16)
        u = field(layer, "up", (M, I), np.uint16)
        for lin, out in ((4, g), (5, u)):
            ref, _ = orc.lora_fwd(b, Wq[base + lin], As[base + lin], Bs[base + lin],
                                  field(layer, "mask", (M, H // 32), np.uint32, lin), s)
            assert rel(f(out), ref) <= TOL
        act = field(layer, "act", (M, I), np.uint16)
        assert ulp_close(act, orc.silu_mul_bf16(g, u))
        h2 = bnd[-1] if layer == cfg.n_layers - 1 else \
            field(layer + 1, "h", (M, H), np.float32).astype(np.float64)
        do, _ = orc.lora_fwd(act, Wq[base + 6], As[base + 6], Bs[base + 6],
                             field(layer, "mask", (M, I // 32), np.uint32, 6), s)
        assert rel(h2 - h1, do) <= TOL


def test_streamed_equals_resident_bitwise_20_steps(ops):
    """The 0.5B-shaped stack (24 layers, seq 512, blocks of 4): resident
    versus streamed through the 2-slot window, 20 Adam steps (lr 2e-4)."""
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=512, H=896, KV=128, I=4864, head_dim=64, n_layers=24)
    wfn, pfn = _fns(0)
    res = StackRun(cfg, 4, False, wfn, pfn)
    stm = StackRun(cfg, 4, True, wfn, pfn)
    assert torch.equal(res.params, stm.params)
    losses = []
    for step in range(20):
        h0 = _h0(cfg, step)
        res.step(step, h0)
        stm.step(step, h0)
        torch.cuda.synchronize()
        assert torch.equal(res.loss, stm.loss), step
        assert torch.equal(res.grads, stm.grads), step
        losses.append(float(res.loss.item()))
    assert ops.device_error() == 0
    for name in ("params", "grads", "adam_m", "adam_v"):
        assert torch.equal(getattr(res, name), getattr(stm, name)), name
    assert all(np.isfinite(losses))
    # the adapters did move
    wfn2, pfn2 = _fns(0)
    fresh = torch.zeros_like(res.params)
    for layer in range(cfg.n_layers):
        for lin, (N, K) in enumerate(cfg.shapes()):
            A, B = pfn2(layer, lin, N, K)
            res.param(layer, lin, "A", fresh).copy_(A)
            res.param(layer, lin, "B", fresh).copy_(B)
    assert not torch.equal(fresh, res.params)


@pytest.mark.parametrize("streamed", [False, True])
def test_graph_replay_equals_eager(ops, streamed):
    """The step captured once as a CUDA graph and replayed with changing step
    numbers (dropout keys and Adam bias corrections read the step from the
    device) gives bitwise the eager call's loss, gradients and state."""
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=256, H=896, KV=128, I=4864, head_dim=64, n_layers=8)
    wfn, pfn = _fns(3)
    eager = StackRun(cfg, 2, streamed, wfn, pfn)
    wfn, pfn = _fns(3)
    graphed = StackRun(cfg, 2, streamed, wfn, pfn)
    cs = torch.cuda.Stream()
    g = graphed.graph(3e-4, cs)
    try:
        for step in (0, 1, 2, 7, 8):
            h0 = _h0(cfg, step)
            eager.step(step, h0, lr=3e-4)
            torch.cuda.synchronize()
            g.step(step, h0, cs)
            cs.synchronize()
            assert torch.equal(eager.loss, graphed.loss), step
            assert torch.equal(eager.grads, graphed.grads), step
    finally:
        g.close()
    for name in ("params", "adam_m", "adam_v"):
        assert torch.equal(getattr(eager, name), getattr(graphed, name)), name
    assert ops.device_error() == 0


def test_stream_block_h2d(ops):
    n = 3 * 2 ** 20 + 4096
    src = torch.randint(0, 255, (n,), dtype=torch.uint8).pin_memory()
    dst = torch.zeros(n, dtype=torch.uint8, device=dev())
    cs = torch.cuda.Stream()
    done = torch.cuda.Event()
    done.record(cs)  # materialise the event handle
    ops.stream_block_h2d(src, dst, copy_stream=cs, done_event=done.cuda_event)
    done.synchronize()
    assert torch.equal(dst.cpu(), src)
    pageable = torch.zeros(4096, dtype=torch.uint8)
    with pytest.raises(ops.WsError) as e:
        ops.stream_block_h2d(pageable, dst)
    assert e.value.status == -8


def test_backward_local_parity(ops, orc):
    """Each backward operation of one layer against the oracle, fed the GPU's
    own inputs (saved activations, the upstream gradient and the workspace's
    intermediate gradients): the linears' input gradients within 1e-4 (fp32
    outputs) and their adapter gradients within TOL, the SwiGLU and repeat
    backward within one bf16 ulp, the RMSNorm backward with its residual
    within 1e-5, the bf16 casts exact; and the forward's residual add exact."""
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=256, H=896, KV=128, I=4864, head_dim=64, n_layers=1)
    wfn, pfn = _fns(6)
    run = StackRun(cfg, 1, False, wfn, pfn)
    M, H, KV, I = cfg.M, cfg.H, cfg.KV, cfg.I
    step = 4
    h0 = _h0(cfg, step)
    saved = torch.empty(run.sizes["saved_layer"], dtype=torch.uint8, device=dev())
    h_out = torch.empty(M * H, device=dev())
    ops.block_forward(cfg, run.dev_weights, 0, 1, run.params, step, h0, h_out, saved, run.workspace)
    dh_out = f32_to_dev(synth.normal_f32(6, "dh_out", (M * H,), 1e-2))
    dh_in = torch.empty_like(dh_out)
    grads = torch.zeros_like(run.params)
    ops.block_backward_recompute(cfg, run.dev_weights, 0, 1, run.params, step, h0, saved, dh_out,
                                 dh_in, grads, run.workspace)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    sv = saved.cpu().numpy()
    ws = run.workspace.cpu().numpy()

    def field(name, shape, dtype, lin=0):
        off = ops.stack_saved_offset(cfg, name, lin)
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return sv[off:off + n].view(dtype).reshape(shape)

    def wk(name, shape, dtype):
        off = ops.stack_workspace_offset(cfg, 1, name)
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return ws[off:off + n].view(dtype).reshape(shape)

    def f(b):
        return synth.bf16_bits_to_f32(b).astype(np.float64)

    def ulp_close(a, b):
        d = np.abs(f(a) - f(b))
        return bool(np.all(d <= np.abs(f(b)) * 2.0 ** -7 + 1e-30) and np.mean(a == b) > 0.99)

    Wq, As, Bs = _oracle_params(orc, cfg, 6)
    s = 2.0 / (1.0 - cfg.p)
    g_all = to_f64(grads)

    def grad(lin, which):
        oA, oB = ops.stack_param_offset(cfg, 0, lin)
        N, K = cfg.shapes()[lin]
        return g_all[oA:oA + 16 * K].reshape(16, K) if which == "A" else \
            g_all[oB:oB + 16 * N].reshape(N, 16)

    def lin_bwd(lin, x_bits, dY_bits):
        N, K = cfg.shapes()[lin]
        mask = field("mask", (M, K // 32), np.uint32, lin)
        dX, dA, dB = orc.lora_bwd(x_bits, Wq[lin], As[lin], Bs[lin], mask, dY_bits, s)
        assert rel(grad(lin, "A"), dA) <= TOL, (lin, "dA")
        assert rel(grad(lin, "B"), dB) <= TOL, (lin, "dB")
        return dX

    h = field("h", (M, H), np.float32).astype(np.float64)
    h1 = field("h1", (M, H), np.float32)
    # forward: the residual add is one exact fp32 add of the bf16 down output
    y_down = wk("yout", (M, H), np.uint16)
    assert np.array_equal(to_f64(h_out).reshape(M, H).astype(np.float32),
                          h1 + synth.bf16_bits_to_f32(y_down))
    # down: dY = bf16(dh_out)
    dY_down = orc.f64_to_bf16(to_f64(dh_out)).reshape(M, H)
    dact = wk("dact", (M, I), np.float32)
    assert rel(dact, lin_bwd(6, field("act", (M, I), np.uint16), dY_down)) <= 1e-4
    # SwiGLU backward
    g = field("gate", (M, I), np.uint16)
    u = field("up", (M, I), np.uint16)
    dg_ref, du_ref = orc.silu_mul_bwd(dact.astype(np.float64), f(g), f(u))
    dg = wk("dg", (M, I), np.uint16)
    du = wk("du", (M, I), np.uint16)
    assert ulp_close(dg, orc.f64_to_bf16(dg_ref).reshape(M, I))
    assert ulp_close(du, orc.f64_to_bf16(du_ref).reshape(M, I))
    # gate and up: their input gradients summed
    b_in = field("b", (M, H), np.uint16)
    db = wk("db", (M, H), np.float32)
    assert rel(db, lin_bwd(4, b_in, dg) + lin_bwd(5, b_in, du)) <= 1e-4
    # RMSNorm 2 backward plus the residual's pass-through
    dh1 = wk("dh1", (M, H), np.float32)
    ref = orc.rmsnorm_bwd(h1.astype(np.float64), field("rstd2", (M,), np.float32), db,
                          dx=to_f64(dh_out).reshape(M, H))
    assert rel(dh1, ref) <= 1e-5
    # o: dY = bf16(dh1), exactly
    y1 = wk("y1", (M, H), np.uint16)
    assert np.array_equal(y1, orc.f64_to_bf16(dh1.astype(np.float64)).reshape(M, H))
    dvr = wk("dvr", (M, H), np.float32)
    assert rel(dvr, lin_bwd(3, field("vr", (M, H), np.uint16), y1)) <= 1e-4
    # repeat backward: the rep query heads of each kv head summed, bf16
    dv = wk("dv", (M, KV), np.uint16)
    assert ulp_close(dv, orc.f64_to_bf16(orc.repeat_kv_bwd(dvr.astype(np.float64), KV,
                                                            cfg.head_dim, round_bf16=False)).reshape(M, KV))
    # v
    da = wk("da", (M, H), np.float32)
    assert rel(da, lin_bwd(2, field("a", (M, H), np.uint16), dv)) <= 1e-4
    # RMSNorm 1 backward plus the residual: the block input's gradient
    ref = orc.rmsnorm_bwd(h, field("rstd1", (M,), np.float32), da, dx=dh1.astype(np.float64))
    assert rel(to_f64(dh_in).reshape(M, H), ref) <= 1e-5
    # q and k: exactly zero
    for lin in (0, 1):
        assert np.all(grad(lin, "A") == 0) and np.all(grad(lin, "B") == 0)
