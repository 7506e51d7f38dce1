"""Pins for the oracle's causal attention core (CPU only).

The attention core is scaled dot-product attention (Vaswani et al., 2017),
causal, with grouped kv heads: query head h reads kv head h // (nh / nkv),
the order in which a transformer repeats its kv heads.  The research page
"Poros" says the learning problem is unchanged by streaming and the model
keeps its own attention; the pages print no formula for it, so the oracle
is this textbook definition written out.

Pins (none re-types the oracle's formula):
- q = 0: every visible key gets the same weight, so o_i is the running mean
  of v over the sequence so far and lse_i = log(i + 1) (closed form);
- the first token of every sequence sees only itself: o_0 = v_0,
  lse_0 = q_0.k_0 / sqrt(d) (pins the 1/sqrt(d) scale and the sequence cut);
- adding one vector c to every key shifts each row's scores by a constant,
  which the softmax removes: o unchanged, lse shifted by q_i.c / sqrt(d);
- causality: changing token t changes no output row before t and nothing in
  another sequence;
- grouped heads equal the same attention with k, v repeated head by head
  (numpy's repeat gives the order h // rep);
- one dominant key: o_i equals that key's value up to exp(-40);
- the backward against central differences of <dO, o>, and two identities
  of the softmax Jacobian: the rows of ds sum to zero, so dk summed over the
  tokens of a sequence vanishes, and the rows of p sum to one, so dv summed
  over tokens equals dO summed over tokens and the sharing query heads.
"""
import numpy as np
import pytest

from weight_streaming_nf4_gb300 import synth


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def test_zero_queries_give_running_mean(orc):
    n_seq, S, nh, nkv, d = 2, 7, 4, 2, 8
    M = n_seq * S
    q = np.zeros((M, nh * d))
    k, v = _rand(1, M, nkv * d), _rand(2, M, nkv * d)
    o, lse = orc.attention_fwd(q, k, v, n_seq, d, want_lse=True)
    for b in range(n_seq):
        for i in range(S):
            t = b * S + i
            for h in range(nh):
                g = h // (nh // nkv)
                mean = v[b * S:t + 1, g * d:(g + 1) * d].mean(axis=0)
                np.testing.assert_allclose(o[t, h * d:(h + 1) * d], mean, rtol=1e-13, atol=1e-14)
                assert abs(lse[h, t] - np.log(i + 1)) < 1e-13


def test_first_token_sees_itself(orc):
    n_seq, S, nh, nkv, d = 3, 5, 2, 1, 16
    M = n_seq * S
    q, k, v = _rand(3, M, nh * d), _rand(4, M, nkv * d), _rand(5, M, nkv * d)
    o, lse = orc.attention_fwd(q, k, v, n_seq, d, want_lse=True)
    for b in range(n_seq):
        t = b * S
        for h in range(nh):
            np.testing.assert_array_equal(o[t, h * d:(h + 1) * d], v[t, :d])
            expect = float(q[t, h * d:(h + 1) * d] @ k[t, :d]) / np.sqrt(d)
            assert abs(lse[h, t] - expect) < 1e-12 * max(1.0, abs(expect))


def test_common_key_shift_changes_nothing(orc):
    n_seq, S, nh, nkv, d = 1, 9, 4, 2, 8
    M = S
    q, k, v = _rand(6, M, nh * d), _rand(7, M, nkv * d), _rand(8, M, nkv * d)
    c = _rand(9, nkv * d)
    o, lse = orc.attention_fwd(q, k, v, n_seq, d, want_lse=True)
    o2, lse2 = orc.attention_fwd(q, k + c[None, :], v, n_seq, d, want_lse=True)
    np.testing.assert_allclose(o2, o, rtol=1e-11, atol=1e-12)
    for h in range(nh):
        g = h // (nh // nkv)
        shift = q[:, h * d:(h + 1) * d] @ c[g * d:(g + 1) * d] / np.sqrt(d)
        np.testing.assert_allclose(lse2[h] - lse[h], shift, rtol=1e-10, atol=1e-11)


def test_causal_and_sequence_independent(orc):
    n_seq, S, nh, nkv, d = 2, 6, 2, 2, 8
    M = n_seq * S
    q, k, v = _rand(10, M, nh * d), _rand(11, M, nkv * d), _rand(12, M, nkv * d)
    o = orc.attention_fwd(q, k, v, n_seq, d)
    for t in [0, 3, 5, 6, 9]:
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[t] += 1.0
        k2[t] -= 0.5
        v2[t] *= 3.0
        o2 = orc.attention_fwd(q2, k2, v2, n_seq, d)
        b = t // S
        changed = np.any(o2 != o, axis=1)
        assert not changed[:t].any()                 # earlier rows, and the earlier sequence
        assert not changed[(b + 1) * S:].any()       # later sequences
        assert changed[t:(b + 1) * S].all()          # rows that see token t


def test_grouped_heads_equal_repeated_kv(orc):
    n_seq, S, nh, nkv, d = 1, 8, 6, 2, 8
    M = S
    rep = nh // nkv
    q, k, v = _rand(13, M, nh * d), _rand(14, M, nkv * d), _rand(15, M, nkv * d)
    kr = np.repeat(k.reshape(M, nkv, d), rep, axis=1).reshape(M, nh * d)
    vr = np.repeat(v.reshape(M, nkv, d), rep, axis=1).reshape(M, nh * d)
    np.testing.assert_array_equal(orc.attention_fwd(q, k, v, n_seq, d),
                                  orc.attention_fwd(q, kr, vr, n_seq, d))
    dO = _rand(16, M, nh * d)
    dq, dk, dv = orc.attention_bwd(q, k, v, dO, n_seq, d)
    dqr, dkr, dvr = orc.attention_bwd(q, kr, vr, dO, n_seq, d)
    np.testing.assert_allclose(dq, dqr, rtol=1e-12, atol=1e-13)
    # the shared kv head collects the gradients of the query heads reading it
    np.testing.assert_allclose(dk, dkr.reshape(M, nkv, rep, d).sum(axis=2).reshape(M, nkv * d),
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dvr.reshape(M, nkv, rep, d).sum(axis=2).reshape(M, nkv * d),
                               rtol=1e-12, atol=1e-13)


def test_one_dominant_key(orc):
    S, d = 6, 16
    target = 2
    alpha = np.sqrt(40.0 * np.sqrt(d))           # score of the target: alpha^2 / sqrt(d) = 40
    q = np.zeros((S, d))
    k = np.zeros((S, d))
    q[4, 0] = alpha
    k[target, 0] = alpha
    v = _rand(17, S, d)
    o = orc.attention_fwd(q, k, v, 1, d)
    # the other four visible keys score 0: their weight is 4 e^-40 / (1 + 4 e^-40)
    np.testing.assert_allclose(o[4], v[target], rtol=0, atol=1e-15 * 50)


def _fd_check(orc, q, k, v, dO, n_seq, d, arrays, rng, h=1e-5):
    dq, dk, dv = orc.attention_bwd(q, k, v, dO, n_seq, d)
    grads = {"q": dq, "k": dk, "v": dv}
    base = {"q": q, "k": k, "v": v}
    checked = 0
    for name in arrays:
        for _ in range(6):
            pos = tuple(rng.integers(s) for s in base[name].shape)
            ins_p = {n: a.copy() for n, a in base.items()}
            ins_m = {n: a.copy() for n, a in base.items()}
            ins_p[name][pos] += h
            ins_m[name][pos] -= h
            lp = np.sum(dO * orc.attention_fwd(ins_p["q"], ins_p["k"], ins_p["v"], n_seq, d))
            lm = np.sum(dO * orc.attention_fwd(ins_m["q"], ins_m["k"], ins_m["v"], n_seq, d))
            fd = (lp - lm) / (2 * h)
            g = grads[name][pos]
            assert abs(fd - g) <= 1e-7 * max(1.0, abs(g)), (name, pos, fd, g)
            checked += 1
    return checked


def test_backward_finite_differences(orc):
    n_seq, S, nh, nkv, d = 2, 5, 4, 2, 8
    M = n_seq * S
    q, k, v = _rand(18, M, nh * d), _rand(19, M, nkv * d), _rand(20, M, nkv * d)
    dO = _rand(21, M, nh * d)
    assert _fd_check(orc, q, k, v, dO, n_seq, d, ["q", "k", "v"], np.random.default_rng(0)) == 18


def test_backward_softmax_identities(orc):
    n_seq, S, nh, nkv, d = 2, 9, 6, 2, 8
    M = n_seq * S
    rep = nh // nkv
    q, k, v = _rand(22, M, nh * d), _rand(23, M, nkv * d), _rand(24, M, nkv * d)
    dO = _rand(25, M, nh * d)
    dq, dk, dv = orc.attention_bwd(q, k, v, dO, n_seq, d)
    for b in range(n_seq):
        rows = slice(b * S, (b + 1) * S)
        np.testing.assert_allclose(dk[rows].sum(axis=0), 0.0, atol=1e-12)
        dO_sum = dO[rows].reshape(S, nkv, rep, d).sum(axis=(0, 2)).reshape(nkv * d)
        np.testing.assert_allclose(dv[rows].sum(axis=0), dO_sum, rtol=1e-12, atol=1e-12)


def test_stack_with_attention_finite_differences(orc):
    """The stack with the attention core in the exact mode: every adapter,
    q and k included, against central differences of the loss."""
    cfg = orc.StackCfg(M=6, H=64, KV=32, I=128, head_dim=16, n_layers=2, r=2, p=0.25,
                       round_bf16=False, attn=1)
    Wq, A, B = [], [], []
    for l in range(cfg.n_layers):
        for li, (N, K) in enumerate(cfg.shapes()):
            W, a, b = synth.stack_weights(0, l, orc.LIN_NAMES[li], N, K, cfg.r)
            codes, absmax = orc.quantize_nf4(W)
            Wq.append(orc.dequant_nf4(codes, absmax))
            A.append(a)
            B.append(b * 10.0)
    h0 = synth.stack_h0(0, 0, cfg.M, cfg.H).astype(np.float64)
    loss, _, dA, dB = orc.stack_fwd_bwd(cfg, 3, Wq, A, B, h0)
    rng = np.random.default_rng(1)
    h = 2.0 ** -15
    for li in range(7):
        for layer in [0, 1]:
            idx = layer * 7 + li
            which = (li + layer) % 2
            arr = A if which == 0 else B
            grad = dA if which == 0 else dB
            pos = tuple(rng.integers(s) for s in arr[idx].shape)
            ap, am = [a.copy() for a in arr], [a.copy() for a in arr]
            ap[idx][pos] += h
            am[idx][pos] -= h
            args_p = (ap, B) if which == 0 else (A, ap)
            args_m = (am, B) if which == 0 else (A, am)
            lp = orc.stack_fwd_bwd(cfg, 3, Wq, *args_p, h0, backward=False)[0]
            lm = orc.stack_fwd_bwd(cfg, 3, Wq, *args_m, h0, backward=False)[0]
            fd = (lp - lm) / (float(ap[idx][pos]) - float(am[idx][pos]))
            g = grad[idx][pos]
            assert abs(fd - g) <= 2e-6 * max(abs(g), 1e-6) + 1e-9, (li, layer, which, fd, g)
    # q and k now carry gradient
    for layer in [0, 1]:
        for li in [0, 1]:
            assert np.any(dB[layer * 7 + li] != 0)


@pytest.mark.parametrize("attn", [0, 1])
def test_stack_recompute_same_keys(orc, attn):
    cfg = orc.StackCfg(M=5, H=64, KV=32, I=128, head_dim=16, n_layers=1, r=2, p=0.1, attn=attn)
    Wq, A, B = [], [], []
    for li, (N, K) in enumerate(cfg.shapes()):
        W, a, b = synth.stack_weights(2, 0, orc.LIN_NAMES[li], N, K, cfg.r)
        codes, absmax = orc.quantize_nf4(W)
        Wq.append(orc.dequant_nf4(codes, absmax))
        A.append(a)
        B.append(b)
    h0 = synth.stack_h0(2, 0, cfg.M, cfg.H).astype(np.float64)
    r1 = orc.stack_fwd_bwd(cfg, 4, Wq, A, B, h0)
    r2 = orc.stack_fwd_bwd(cfg, 4, Wq, A, B, h0)
    assert r1[0] == r2[0]
    np.testing.assert_array_equal(r1[1], r2[1])
