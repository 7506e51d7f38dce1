"""GPU tests of the block engine (a6-a9): block forward / backward with
recompute, the streamed training step, and the pinned-host block copy.

- The recompute (forward rerun from the block-boundary activation with the
  same Philox keys) reproduces the kept intermediates bit for bit, so the
  recomputed backward equals the resident backward exactly (research page
  "Poros": "The recomputed forward reproduces the original exactly, down to
  the bit").
- A streamed run equals a resident run bitwise on loss, gradients,
  parameters and both Adam moments over 20 steps (research page "Poros":
  loss, adapter weights, gradient norms and optimizer state "match a
  fully-resident run exactly ... checked with torch.equal").
- One step of a 2-layer stack matches the fp64 oracle within TOL.
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


def test_one_step_matches_oracle(ops, orc):
    """Loss and every adapter gradient of one step of a 2-layer stack with the
    0.5B widths (H 896, kv 128, I 4864, head_dim 64), against the oracle."""
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=128, H=896, KV=128, I=4864, head_dim=64, n_layers=2)
    wfn, pfn = _fns(2)
    run = StackRun(cfg, 2, False, wfn, pfn)
    step = 5
    run.step(step, _h0(cfg, step), lr=0.0)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    names = ("q", "k", "v", "o", "gate", "up", "down")
    Wq, As, Bs = [], [], []
    for layer in range(cfg.n_layers):
        for lin, (N, K) in enumerate(cfg.shapes()):
            W, A, B = synth.stack_weights(2, layer, names[lin], N, K)
            Wq.append(orc.dequant_nf4(*orc.quantize_nf4(W)))
            As.append(A)
            Bs.append(B)
    ocfg = orc.StackCfg(M=cfg.M, H=cfg.H, KV=cfg.KV, I=cfg.I, head_dim=cfg.head_dim,
                        n_layers=cfg.n_layers, p=cfg.p)
    h0 = synth.stack_h0(cfg.seed, step, cfg.M, cfg.H).astype(np.float64)
    loss, _, dA, dB = orc.stack_fwd_bwd(ocfg, step, Wq, As, Bs, h0)
    assert abs(float(run.loss.item()) - loss) <= 1e-4 * abs(loss)
    for layer in range(cfg.n_layers):
        for lin in range(7):
            gA = to_f64(run.param(layer, lin, "A", run.grads))
            gB = to_f64(run.param(layer, lin, "B", run.grads))
            i = layer * 7 + lin
            if lin in (0, 1):
                assert np.all(gA == 0) and np.all(gB == 0)
                continue
            assert rel(gA, dA[i]) <= TOL, (layer, names[lin], "A", rel(gA, dA[i]))
            assert rel(gB, dB[i]) <= TOL, (layer, names[lin], "B", rel(gB, dB[i]))


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
