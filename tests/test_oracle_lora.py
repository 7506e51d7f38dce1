"""Pins for the oracle's NF4-LoRA linear (CPU only).

Each linear computes y = x W'^T + (alpha/r) B A dropout(x) with the frozen
W' = dequant(NF4(W)); the backward produces only dX, dA and dB because
frozen weights are never differentiated (research page "Poros": the backward
"propagates gradients only to the adapters and block inputs").  With
inverted dropout the (1-p)^-1 factor is folded into scale = (alpha/r)/(1-p).

Pins: a literal triple loop on tiny shapes, numpy float64 matmul (a library
routine) on moderate shapes, exactness of the gradients from the forward's
linearity (unit inputs), central differences, and the special cases p = 0,
A = 0, B = 0.
"""
import numpy as np

from weight_streaming_nf4_gb300 import synth


def _f(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def _mask_dense(bits, M, K):
    m = np.zeros((M, K), np.float64)
    for i in range(M):
        for k in range(K):
            m[i, k] = (int(bits[i, k // 32]) >> (k % 32)) & 1
    return m


def _setup(orc, M, N, K, r, p=0.1, tag="t"):
    d = synth.linear_inputs(0, M, N, K, r, tag=tag)
    codes, absmax = orc.quantize_nf4(d["W"])
    Wq = orc.dequant_nf4(codes, absmax)
    mask = orc.dropout_mask(0, 0, 0, 0, 0, p, M, K)
    scale = (32.0 / r) / (1.0 - p)
    return d, Wq, mask, scale


def test_fwd_bwd_triple_loop(orc):
    M, N, K, r = 3, 5, 64, 2
    d, Wq, mask, s = _setup(orc, M, N, K, r)
    x, W, A, B, dY = _f(d["x"]), _f(Wq), d["A"].astype(float), d["B"].astype(float), _f(d["dY"])
    md = _mask_dense(mask, M, K)
    y = np.zeros((M, N))
    U = np.zeros((M, r))
    for m in range(M):
        for j in range(r):
            for k in range(K):
                U[m, j] += md[m, k] * x[m, k] * A[j, k]
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += x[m, k] * W[n, k]
            for j in range(r):
                acc += s * U[m, j] * B[n, j]
            y[m, n] = acc
    yo, Uo = orc.lora_fwd(d["x"], Wq, d["A"], d["B"], mask, s)
    np.testing.assert_allclose(yo, y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Uo, U, rtol=1e-12, atol=1e-14)
    G = np.zeros((M, r))
    for m in range(M):
        for j in range(r):
            for n in range(N):
                G[m, j] += dY[m, n] * B[n, j]
    dX = np.zeros((M, K))
    for m in range(M):
        for k in range(K):
            acc = 0.0
            for n in range(N):
                acc += dY[m, n] * W[n, k]
            for j in range(r):
                acc += s * md[m, k] * G[m, j] * A[j, k]
            dX[m, k] = acc
    dA = np.zeros((r, K))
    for j in range(r):
        for k in range(K):
            for m in range(M):
                dA[j, k] += s * G[m, j] * md[m, k] * x[m, k]
    dB = np.zeros((N, r))
    for n in range(N):
        for j in range(r):
            for m in range(M):
                dB[n, j] += s * dY[m, n] * U[m, j]
    dXo, dAo, dBo = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], mask, d["dY"], s)
    np.testing.assert_allclose(dXo, dX, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dAo, dA, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dBo, dB, rtol=1e-12, atol=1e-14)


def test_against_numpy_matmul(orc):
    M, N, K, r = 40, 96, 192, 16
    d, Wq, mask, s = _setup(orc, M, N, K, r)
    x, W, A, B, dY = _f(d["x"]), _f(Wq), d["A"].astype(float), d["B"].astype(float), _f(d["dY"])
    md = _mask_dense(mask, M, K)
    xm = md * x
    U = xm @ A.T
    y = x @ W.T + s * U @ B.T
    yo, Uo = orc.lora_fwd(d["x"], Wq, d["A"], d["B"], mask, s)
    np.testing.assert_allclose(yo, y, rtol=1e-10, atol=1e-12)
    G = dY @ B
    dX = dY @ W + s * md * (G @ A)
    dA = s * G.T @ xm
    dB = s * dY.T @ U
    dXo, dAo, dBo = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], mask, d["dY"], s)
    np.testing.assert_allclose(dXo, dX, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dAo, dA, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dBo, dB, rtol=1e-10, atol=1e-12)
    # row subsets give the same rows
    rows = np.array([39, 0, 17])
    ys, _ = orc.lora_fwd(d["x"], Wq, d["A"], d["B"], mask, s, rows=rows)
    np.testing.assert_array_equal(ys, yo[rows])
    dXs, _, _ = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], mask, d["dY"], s, rows=rows)
    np.testing.assert_array_equal(dXs, dXo[rows])


def _loss(orc, x, Wq, A, B, mask, s, dY):
    y, _ = orc.lora_fwd(x, Wq, A, B, mask, s)
    return float(np.sum(_f(dY) * y))


def test_gradients_from_forward_linearity(orc):
    """L = <dY, y> is linear in x, in A and in B separately, so each gradient
    entry equals L evaluated at a unit input (minus the value at zero)."""
    M, N, K, r = 4, 8, 64, 2
    d, Wq, mask, s = _setup(orc, M, N, K, r, tag="lin")
    dX, dA, dB = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], mask, d["dY"], s)
    one = synth.to_bf16_bits(np.array([1.0]))[0]
    rng = np.random.default_rng(0)
    for _ in range(12):
        m, k = rng.integers(M), rng.integers(K)
        xe = np.zeros((M, K), np.uint16)
        xe[m, k] = one
        np.testing.assert_allclose(_loss(orc, xe, Wq, d["A"], d["B"], mask, s, d["dY"]), dX[m, k],
                                   rtol=1e-12, atol=1e-13)
    L0A = _loss(orc, d["x"], Wq, np.zeros_like(d["A"]), d["B"], mask, s, d["dY"])
    for _ in range(8):
        j, k = rng.integers(r), rng.integers(K)
        Ae = np.zeros_like(d["A"])
        Ae[j, k] = 1.0
        got = _loss(orc, d["x"], Wq, Ae, d["B"], mask, s, d["dY"]) - L0A
        np.testing.assert_allclose(got, dA[j, k], rtol=1e-9, atol=1e-12)
    L0B = _loss(orc, d["x"], Wq, d["A"], np.zeros_like(d["B"]), mask, s, d["dY"])
    for _ in range(8):
        n, j = rng.integers(N), rng.integers(r)
        Be = np.zeros_like(d["B"])
        Be[n, j] = 1.0
        got = _loss(orc, d["x"], Wq, d["A"], Be, mask, s, d["dY"]) - L0B
        np.testing.assert_allclose(got, dB[n, j], rtol=1e-9, atol=1e-12)


def test_central_differences(orc):
    M, N, K, r = 4, 8, 64, 2
    d, Wq, mask, s = _setup(orc, M, N, K, r, tag="fd")
    _, dA, dB = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], mask, d["dY"], s)
    h = 2.0 ** -12
    for (j, k) in [(0, 3), (1, 40), (0, 63)]:
        Ap, Am = d["A"].copy(), d["A"].copy()
        Ap[j, k] += h
        Am[j, k] -= h
        fd = (_loss(orc, d["x"], Wq, Ap, d["B"], mask, s, d["dY"])
              - _loss(orc, d["x"], Wq, Am, d["B"], mask, s, d["dY"])) / (float(Ap[j, k]) - float(Am[j, k]))
        np.testing.assert_allclose(fd, dA[j, k], rtol=1e-6, atol=1e-9)
    for (n, j) in [(0, 0), (7, 1), (3, 1)]:
        Bp, Bm = d["B"].copy(), d["B"].copy()
        Bp[n, j] += h
        Bm[n, j] -= h
        fd = (_loss(orc, d["x"], Wq, d["A"], Bp, mask, s, d["dY"])
              - _loss(orc, d["x"], Wq, d["A"], Bm, mask, s, d["dY"])) / (float(Bp[n, j]) - float(Bm[n, j]))
        np.testing.assert_allclose(fd, dB[n, j], rtol=1e-6, atol=1e-9)


def test_special_cases(orc):
    M, N, K, r = 8, 16, 128, 16
    d, Wq, mask, s = _setup(orc, M, N, K, r, p=0.0, tag="sp")
    assert np.all(mask == 0xFFFFFFFF)
    x, W = _f(d["x"]), _f(Wq)
    # A = 0: pure frozen-base product
    y, U = orc.lora_fwd(d["x"], Wq, np.zeros_like(d["A"]), d["B"], mask, s)
    np.testing.assert_allclose(y, x @ W.T, rtol=1e-12, atol=1e-13)
    assert np.all(U == 0)
    # B = 0: no adapter contribution, zero dA, dX = dY W'
    dX, dA, dB = orc.lora_bwd(d["x"], Wq, d["A"], np.zeros_like(d["B"]), mask, d["dY"], s)
    assert np.all(dA == 0)
    np.testing.assert_allclose(dX, _f(d["dY"]) @ W, rtol=1e-12, atol=1e-13)
    # unit rows of x pick out columns of W' exactly
    xe = np.zeros((M, K), np.uint16)
    ks = [0, 5, 64, 127, 1, 2, 3, 100]
    for m, k in enumerate(ks):
        xe[m, k] = synth.to_bf16_bits(np.array([1.0]))[0]
    y, _ = orc.lora_fwd(xe, Wq, d["A"], np.zeros_like(d["B"]), mask, s)
    for m, k in enumerate(ks):
        assert np.array_equal(y[m], W[:, k])
