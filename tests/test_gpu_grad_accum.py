"""Gradient accumulation on the GPU: a step over several micro-batches, each
with its own input and its own dropout keys (the micro-batch index is part
of the Philox counter).

The pages gate accumulation at 2 and 4 micro-batches and refuse the
block-major order combined with dropout, because their sequential RNG would
then be consumed in another order (research page "Poros", block-major and
parity-gate paragraphs).  With counter-based keys the order is free, so here
both orders must give the resident run's step bit for bit: loss, gradients,
parameters and both Adam moments, over 20 steps of the 0.5B-shaped stack.
One accumulated step of a small stack also matches the oracle, whose
micro-batch keys and loss averaging are pinned on the CPU.
"""
import numpy as np
import pytest
import torch

from gpu_util import f32_to_dev, rel, to_f64
from test_gpu_stack import STACK_TOL, _fns, _oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _h0s(cfg, step, n_micro):
    from weight_streaming_nf4_gb300 import synth
    return f32_to_dev(np.concatenate(
        [synth.stack_h0(cfg.seed, 1000 * step + mb, cfg.M, cfg.H).ravel() for mb in range(n_micro)]))


@pytest.mark.parametrize("n_micro", [2, 4])
def test_accumulated_steps_streamed_equal_resident(ops, n_micro):
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=512, H=896, KV=128, I=4864, head_dim=64, n_layers=24)
    wfn, pfn = _fns(0)
    res = StackRun(cfg, 4, False, wfn, pfn, n_micro=n_micro)
    mbm = StackRun(cfg, 4, True, wfn, pfn, image_from=res, n_micro=n_micro,
                   order=ops.GA_MICROBATCH_MAJOR)
    blm = StackRun(cfg, 4, True, wfn, pfn, image_from=res, n_micro=n_micro,
                   order=ops.GA_BLOCK_MAJOR)
    runs = (res, mbm, blm)
    for step in range(20):
        h0 = _h0s(cfg, step, n_micro)
        for r in runs:
            r.step(step, h0)
        torch.cuda.synchronize()
        for r in runs[1:]:
            assert torch.equal(res.loss, r.loss), (step, r.order)
            assert torch.equal(res.grads, r.grads), (step, r.order)
    assert ops.device_error() == 0
    for r in runs[1:]:
        for name in ("params", "grads", "adam_m", "adam_v"):
            assert torch.equal(getattr(res, name), getattr(r, name)), (name, r.order)
    assert np.isfinite(float(res.loss.item()))


def test_accumulation_is_not_a_repeat_of_one_micro_batch(ops):
    """The micro-batches differ (inputs and masks): the accumulated gradient
    is not n times one micro-batch's gradient, and one micro-batch through
    the accumulating step equals the plain step bitwise."""
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=128, H=256, KV=64, I=512, head_dim=32, n_layers=2)
    wfn, pfn = _fns(5)
    one = StackRun(cfg, 1, False, wfn, pfn)
    plain = StackRun(cfg, 1, False, wfn, pfn)
    two = StackRun(cfg, 1, False, wfn, pfn, n_micro=2)
    h0 = _h0s(cfg, 3, 2)
    M, H = cfg.M, cfg.H
    one.step(3, h0[:M * H], lr=0.0)
    from weight_streaming_nf4_gb300 import ops as o
    o.stack_train_step(cfg, 1, False, plain.c, 3, h0[:M * H], 0.0)  # opts = None
    two.step(3, h0, lr=0.0)
    torch.cuda.synchronize()
    assert torch.equal(one.grads, plain.grads) and torch.equal(one.loss, plain.loss)
    assert not torch.equal(two.grads, one.grads)
    assert not torch.allclose(two.grads, 2 * one.grads, rtol=1e-3, atol=0)


def test_accumulated_step_matches_oracle(ops, orc):
    """Two micro-batches through a 2-layer stack with the 0.5B widths: the
    step loss (mean over micro-batches) and every adapter gradient (sum over
    micro-batches) against the oracle."""
    from weight_streaming_nf4_gb300 import synth
    from weight_streaming_nf4_gb300.stack import StackRun
    cfg = ops.StackCfg(M=128, H=896, KV=128, I=4864, head_dim=64, n_layers=2)
    wfn, pfn = _fns(7)
    run = StackRun(cfg, 2, True, wfn, pfn, n_micro=2, order=ops.GA_BLOCK_MAJOR)
    step = 6
    run.step(step, _h0s(cfg, step, 2), lr=0.0)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    Wq, As, Bs = _oracle_params(orc, cfg, 7)
    ocfg = orc.StackCfg(M=cfg.M, H=cfg.H, KV=cfg.KV, I=cfg.I, head_dim=cfg.head_dim,
                        n_layers=cfg.n_layers, p=cfg.p)
    loss, dA, dB = 0.0, None, None
    for mb in range(2):
        h0 = synth.stack_h0(cfg.seed, 1000 * step + mb, cfg.M, cfg.H).astype(np.float64)
        l, _, a, b = orc.stack_fwd_bwd(ocfg, step, Wq, As, Bs, h0, microbatch=mb, n_micro=2)
        loss += l
        dA = a if dA is None else [x + y for x, y in zip(dA, a)]
        dB = b if dB is None else [x + y for x, y in zip(dB, b)]
    assert abs(float(run.loss.item()) - loss) <= 1e-4 * abs(loss)
    for layer in range(cfg.n_layers):
        for lin in range(2, 7):
            i = layer * 7 + lin
            assert rel(to_f64(run.param(layer, lin, "A", run.grads)), dA[i]) <= STACK_TOL, (layer, lin)
            assert rel(to_f64(run.param(layer, lin, "B", run.grads)), dB[i]) <= STACK_TOL, (layer, lin)
