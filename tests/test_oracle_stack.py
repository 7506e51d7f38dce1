"""Pins for the oracle's synthetic transformer stack and Adam (CPU only).

The stack is the layer construction the method is measured on, with the
attention core replaced by repeating v across the query heads:
RMSNorm -> q,k,v -> repeat(v) -> o -> residual; RMSNorm -> gate,up ->
SiLU(gate)*up -> down -> residual; loss = 0.5 mean(h_L^2).  Streaming changes
nothing numerically (research page "Poros": the adapter is "the same, bit for
bit"), so the oracle is this plain definition.

Pins: central differences of the loss in the exact mode (no bf16 rounding),
which exercise every backward formula (RMSNorm, SiLU*up, repeat_kv, residual,
loss); a zero-weight stack that must reduce to the identity; recompute with
the same keys reproducing the forward exactly (research page "Poros", "RNG
state capture"); Adam against its closed form for a constant gradient.
"""
import numpy as np

from weight_streaming_nf4_gb300 import synth


def _toy(orc, cfg, seed=0, zero=False):
    Wq, A, B = [], [], []
    for l in range(cfg.n_layers):
        for li, (N, K) in enumerate(cfg.shapes()):
            W, a, b = synth.stack_weights(seed, l, orc.LIN_NAMES[li], N, K, cfg.r)
            if zero:
                W = np.zeros_like(W)
                b = np.zeros_like(b)
            codes, absmax = orc.quantize_nf4(W)
            Wq.append(orc.dequant_nf4(codes, absmax))
            A.append(a)
            # larger B than the default so the adapter paths carry weight
            B.append(b * 10.0)
    return Wq, A, B


def test_stack_finite_differences_exact_mode(orc):
    cfg = orc.StackCfg(M=4, H=64, KV=32, I=128, head_dim=16, n_layers=2, r=2, p=0.25,
                       round_bf16=False)
    Wq, A, B = _toy(orc, cfg)
    h0 = synth.stack_h0(0, 0, cfg.M, cfg.H).astype(np.float64)
    loss, _, dA, dB = orc.stack_fwd_bwd(cfg, 5, Wq, A, B, h0)
    rng = np.random.default_rng(0)
    h = 2.0 ** -15
    checked = 0
    for li in [2, 3, 4, 5, 6]:          # v, o, gate, up, down (q, k are dead)
        for layer in [0, 1]:
            idx = layer * 7 + li
            for _ in range(2):
                which = rng.integers(2)
                arr = A if which == 0 else B
                grad = dA if which == 0 else dB
                pos = tuple(rng.integers(s) for s in arr[idx].shape)
                ap, am = [a.copy() for a in arr], [a.copy() for a in arr]
                ap[idx][pos] += h
                am[idx][pos] -= h
                args_p = (ap, B) if which == 0 else (A, ap)
                args_m = (am, B) if which == 0 else (A, am)
                lp = orc.stack_fwd_bwd(cfg, 5, Wq, *args_p, h0, backward=False)[0]
                lm = orc.stack_fwd_bwd(cfg, 5, Wq, *args_m, h0, backward=False)[0]
                fd = (lp - lm) / (float(ap[idx][pos]) - float(am[idx][pos]))
                g = grad[idx][pos]
                assert abs(fd - g) <= 2e-6 * max(abs(g), 1e-6) + 1e-9, (li, layer, which, fd, g)
                checked += 1
    assert checked == 20
    for layer in [0, 1]:
        for li in [0, 1]:
            assert np.all(dA[layer * 7 + li] == 0) and np.all(dB[layer * 7 + li] == 0)


def test_zero_weights_stack_is_identity(orc):
    cfg = orc.StackCfg(M=4, H=64, KV=32, I=128, head_dim=16, n_layers=2, r=2, p=0.1)
    Wq, A, B = _toy(orc, cfg, zero=True)
    h0 = synth.stack_h0(0, 1, cfg.M, cfg.H).astype(np.float64)
    loss, hL, dA, dB = orc.stack_fwd_bwd(cfg, 1, Wq, A, B, h0)
    assert np.array_equal(hL, h0)
    np.testing.assert_allclose(loss, 0.5 * np.mean(h0 ** 2), rtol=1e-15)
    for a in dA:
        assert np.all(a == 0)


def test_recompute_with_same_keys_is_exact(orc):
    cfg = orc.StackCfg(M=8, H=64, KV=32, I=128, head_dim=16, n_layers=2, r=4, p=0.1)
    Wq, A, B = _toy(orc, cfg)
    h0 = synth.stack_h0(0, 2, cfg.M, cfg.H).astype(np.float64)
    r1 = orc.stack_fwd_bwd(cfg, 2, Wq, A, B, h0)
    r2 = orc.stack_fwd_bwd(cfg, 2, Wq, A, B, h0)
    assert r1[0] == r2[0] and np.array_equal(r1[1], r2[1])
    for a, b in zip(r1[2] + r1[3], r2[2] + r2[3]):
        assert np.array_equal(a, b)
    r3 = orc.stack_fwd_bwd(cfg, 3, Wq, A, B, h0)   # another step draws other masks
    assert r3[0] != r1[0]


def test_adam_constant_gradient_closed_form(orc):
    """With a constant gradient g the bias-corrected moments equal g and g^2
    exactly, so every step moves p by -lr * g / (|g| + eps)."""
    rng = np.random.default_rng(0)
    g = rng.normal(0, 1e-3, 50)
    g[0] = 0.0
    p0 = rng.normal(0, 1, 50)
    p, m, v = p0.copy(), np.zeros(50), np.zeros(50)
    lr, eps = 2e-4, 1e-8
    for t in range(1, 6):
        orc.adam_step(p, g.copy(), m, v, t, lr=lr, eps=eps)
        np.testing.assert_allclose(p, p0 - t * lr * g / (np.abs(g) + eps), rtol=1e-12, atol=1e-15)
    assert p[0] == p0[0]


def test_gradient_accumulation_micro_batches(orc):
    """A step with gradient accumulation over two micro-batches: the step
    loss is the mean of the micro-batch losses and its gradient the sum of
    the micro-batch calls' gradients (central differences of the step loss in
    the exact mode); the micro-batch index enters the dropout keys, and one
    micro-batch reduces to the plain step."""
    cfg = orc.StackCfg(M=4, H=64, KV=32, I=128, head_dim=16, n_layers=1, r=2, p=0.25,
                       round_bf16=False)
    Wq, A, B = _toy(orc, cfg, seed=3)
    h0s = [synth.stack_h0(3, 10 + mb, cfg.M, cfg.H).astype(np.float64) for mb in range(2)]

    def step(Aa, Bb, backward=True):
        tot, gA, gB = 0.0, None, None
        for mb in range(2):
            loss, _, dA, dB = orc.stack_fwd_bwd(cfg, 4, Wq, Aa, Bb, h0s[mb], backward=backward,
                                                microbatch=mb, n_micro=2)
            tot += loss
            if backward:
                gA = dA if gA is None else [x + y for x, y in zip(gA, dA)]
                gB = dB if gB is None else [x + y for x, y in zip(gB, dB)]
        return tot, gA, gB

    _, gA, gB = step(A, B)
    h = 2.0 ** -15
    for li, which, pos in [(2, 0, (1, 5)), (3, 1, (7, 0)), (4, 0, (0, 9)), (6, 1, (3, 1))]:
        arr = A if which == 0 else B
        ap, am = [a.copy() for a in arr], [a.copy() for a in arr]
        ap[li][pos] += h
        am[li][pos] -= h
        lp = step(ap, B, False)[0] if which == 0 else step(A, ap, False)[0]
        lm = step(am, B, False)[0] if which == 0 else step(A, am, False)[0]
        fd = (lp - lm) / (float(ap[li][pos]) - float(am[li][pos]))
        g = (gA if which == 0 else gB)[li][pos]
        assert abs(fd - g) <= 2e-6 * max(abs(g), 1e-6) + 1e-9, (li, which, fd, g)
    # other micro-batch index, other masks: same input, other loss
    l0 = orc.stack_fwd_bwd(cfg, 4, Wq, A, B, h0s[0], backward=False, microbatch=0, n_micro=2)[0]
    l1 = orc.stack_fwd_bwd(cfg, 4, Wq, A, B, h0s[0], backward=False, microbatch=1, n_micro=2)[0]
    assert l0 != l1
    # one micro-batch is the plain step
    r1 = orc.stack_fwd_bwd(cfg, 4, Wq, A, B, h0s[0])
    r2 = orc.stack_fwd_bwd(cfg, 4, Wq, A, B, h0s[0], microbatch=0, n_micro=1)
    assert r1[0] == r2[0] and all(np.array_equal(x, y) for x, y in zip(r1[2], r2[2]))
