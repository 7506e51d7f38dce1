"""GPU parity of the NF4-LoRA linear (quantiser, masks, forward, backward) against the CPU oracle, through
the C ABI.  Integer work (NF4 codes, absmax, dropout bits) must be bit-exact;
floating outputs (y, dX, dA, dB) within the normwise tolerance TOL of the
fp64 oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_bits, bf16_to_dev, dev, f32_to_dev, rel, to_f64

pytestmark = pytest.mark.gpu

P = 0.1


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _linear(ops, orc, M, N, K, tag, seed=0, p=P, layer=0, lin=0, step=0):
    from weight_streaming_nf4_gb300 import synth
    d = synth.linear_inputs(seed, M, N, K, 16, tag=tag)
    codes, absmax = ops.quantize_nf4(bf16_to_dev(d["W"]))
    W = ops.NF4Weight(codes, absmax, N, K)
    key = ops.dropout_key(seed=seed, step=step, layer=layer, linear=lin, p=p)
    return d, W, key


def test_quantize_bit_exact(ops, orc):
    from weight_streaming_nf4_gb300 import synth
    for (N, K, std) in [(512, 512, 0.02), (896, 4864, 0.02), (64, 128, 3.0), (192, 1024, 1e-3)]:
        W = synth.normal_bf16(1, f"q{N}x{K}", (N, K), std)
        W[3, 64:128] = 0                      # an all-zero block
        W[5, 0:64] = W[5, 7]                  # a constant block
        codes, absmax = ops.quantize_nf4(bf16_to_dev(W))
        oc, oa = orc.quantize_nf4(W)
        assert np.array_equal(codes.cpu().numpy(), oc), (N, K)
        assert np.array_equal(absmax.cpu().numpy().view(np.uint32), oa.view(np.uint32)), (N, K)


def test_dropout_mask_bit_exact(ops, orc):
    for (M, N, K, step, layer, lin, p) in [(64, 512, 512, 0, 0, 0, 0.1), (300, 128, 896, 7, 3, 5, 0.1),
                                           (33, 64, 4864, 2, 23, 6, 0.25), (16, 64, 64, 0, 0, 0, 0.0)]:
        d, W, key = _linear(ops, orc, M, N, K, "mask", layer=layer, lin=lin, step=step, p=p)
        _, _, mask = ops.lora_linear_fwd(W, bf16_to_dev(d["x"]), f32_to_dev(d["A"]),
                                         f32_to_dev(d["B"]), key)
        om = orc.dropout_mask(0, step, layer, lin, 0, p, M, K)
        assert np.array_equal(mask.cpu().numpy().view(np.uint32), om), (M, K)


def test_dequant_through_gemm_is_exact(ops, orc):
    """x = unit rows e_k and B = 0: y[m, :] = W'[:, k_m] exactly (one
    non-zero product per output, exact fp32 accumulation, exact bf16 store)."""
    for (M, N, K) in [(128, 512, 512), (256, 768, 1024), (64, 128, 4864)]:
        from weight_streaming_nf4_gb300 import synth
        Wb = synth.normal_bf16(2, f"pin{N}", (N, K), 0.02)
        codes, absmax = ops.quantize_nf4(bf16_to_dev(Wb))
        W = ops.NF4Weight(codes, absmax, N, K)
        rng = np.random.default_rng(N)
        ks = rng.integers(0, K, size=M)
        x = np.zeros((M, K), np.uint16)
        x[np.arange(M), ks] = synth.to_bf16_bits(np.array([1.0]))[0]
        A = np.zeros((16, K), np.float32)
        B = np.zeros((N, 16), np.float32)
        y, _, _ = ops.lora_linear_fwd(W, bf16_to_dev(x), f32_to_dev(A), f32_to_dev(B),
                                      ops.dropout_key(p=0.0))
        Wq = orc.dequant_nf4(*orc.quantize_nf4(Wb))
        assert np.array_equal(bf16_bits(y), Wq[:, ks].T), (M, N, K)


SHAPES = [
    (64, 512, 512),      # the single-linear workload (one tile, M < 128)
    (300, 896, 1088),    # ragged M (3 x 128 - 84), ragged N (3.5 x 256)
    (64, 512, 4096),     # few tiles: deep contraction split across CTAs
    (512, 128, 896),     # narrow N (0.5B k/v shape)
    (200, 4864, 896),    # 0.5B gate shape, ragged M
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_fwd_bwd_parity(ops, orc, M, N, K):
    d, W, key = _linear(ops, orc, M, N, K, f"lin{M}x{N}x{K}", lin=3, layer=2, step=1)
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])
    y, U, mask = ops.lora_linear_fwd(W, x, A, B, key)
    dXb, dA, dB = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY)
    dXf, dA2, dB2 = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX_f32=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    oc, oa = orc.quantize_nf4(d["W"])
    Wq = orc.dequant_nf4(oc, oa)
    om = orc.dropout_mask(0, 1, 2, 3, 0, P, M, K)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), om)
    s = 2.0 / (1.0 - P)
    yo, Uo = orc.lora_fwd(d["x"], Wq, d["A"], d["B"], om, s)
    dXo, dAo, dBo = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], om, d["dY"], s)
    assert rel(to_f64(y), yo) <= TOL
    assert rel(to_f64(U), Uo) <= 1e-5
    assert rel(to_f64(dXb), dXo) <= TOL
    assert rel(to_f64(dXf), dXo) <= 1e-4
    assert rel(to_f64(dA), dAo) <= TOL and rel(to_f64(dB), dBo) <= TOL
    # the two backward calls share every reduction: identical gradients
    assert torch.equal(dA, dA2) and torch.equal(dB, dB2)
    # elementwise: y within one bf16 ulp (+ fp32 accumulation slack) of the oracle
    yf = to_f64(y)
    assert np.all(np.abs(yf - yo) <= np.abs(yo) * 2.0 ** -8 + 1e-3 * np.abs(yo).max())


def test_bwd_regenerates_masks_and_is_deterministic(ops, orc):
    M, N, K = 256, 512, 1024
    d, W, key = _linear(ops, orc, M, N, K, "det", lin=5, layer=1, step=4)
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])
    y1, U1, m1 = ops.lora_linear_fwd(W, x, A, B, key)
    y2, U2, _ = ops.lora_linear_fwd(W, x, A, B, key, keep_mask=False)
    assert torch.equal(y1, y2) and torch.equal(U1, U2)
    r1 = ops.lora_linear_bwd(W, x, A, B, key, U1, m1, dY, dX_f32=True)
    r2 = ops.lora_linear_bwd(W, x, A, B, key, U1, None, dY, dX_f32=True)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_dx_accumulate(ops, orc):
    M, N, K = 128, 256, 512
    d, W, key = _linear(ops, orc, M, N, K, "acc")
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])
    _, U, mask = ops.lora_linear_fwd(W, x, A, B, key)
    dX, _, _ = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX_f32=True)
    base = torch.randn(M, K, device=dev())
    acc = base.clone()
    ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX=acc, accumulate=True)
    assert torch.equal(acc, base + dX)


def test_grad_accumulate(ops, orc):
    """WS_ACC_GRADS adds dA and dB into the given gradients: one fp32 add of
    the fresh gradient, bitwise; the input gradient is unaffected."""
    M, N, K = 192, 512, 1024
    d, W, key = _linear(ops, orc, M, N, K, "gacc", lin=2)
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])
    _, U, mask = ops.lora_linear_fwd(W, x, A, B, key)
    dX, dA, dB = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX_f32=True)
    a0 = torch.randn_like(dA)
    b0 = torch.randn_like(dB)
    a, b = a0.clone(), b0.clone()
    dX2, _, _ = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX_f32=True, dA=a, dB=b,
                                    grad_accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(a, a0 + dA) and torch.equal(b, b0 + dB)
    assert torch.equal(dX2, dX)


@pytest.mark.parametrize("M,N,K,lin", [(512, 18944, 3584, 4), (512, 3584, 18944, 6),
                                        (2048, 512, 3584, 2)])
def test_full_size_sampled_rows(ops, orc, M, N, K, lin):
    """7B-layer shapes at the benchmark's launch configuration; the oracle
    evaluates a sample of rows of y and dX and the full dA, dB."""
    d, W, key = _linear(ops, orc, M, N, K, f"full{lin}", lin=lin)
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])
    y, U, mask = ops.lora_linear_fwd(W, x, A, B, key)
    dX, dA, dB = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    oc, oa = orc.quantize_nf4(d["W"])
    assert np.array_equal(W.codes.cpu().numpy(), oc)
    Wq = orc.dequant_nf4(oc, oa)
    om = orc.dropout_mask(0, 0, 0, lin, 0, P, M, K)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), om)
    rows = np.array([0, 1, 127, 128, 255, M // 2 + 3, M - 1])
    s = 2.0 / (1.0 - P)
    yo, _ = orc.lora_fwd(d["x"], Wq, d["A"], d["B"], om, s, rows=rows)
    dXo, dAo, dBo = orc.lora_bwd(d["x"], Wq, d["A"], d["B"], om, d["dY"], s, rows=rows)
    assert rel(to_f64(y)[rows], yo) <= TOL
    assert rel(to_f64(dX)[rows], dXo) <= TOL
    assert rel(to_f64(dA), dAo) <= TOL and rel(to_f64(dB), dBo) <= TOL


@pytest.mark.parametrize("M,N,K", [(64, 512, 512), (300, 896, 1088), (512, 3584, 3584)])
def test_nf4_matmul_alone(ops, orc, M, N, K):
    """The frozen product without adapter: x W'^T and dY W'."""
    d, W, _ = _linear(ops, orc, M, N, K, f"mm{M}")
    Wq = orc.dequant_nf4(*orc.quantize_nf4(d["W"]))
    y = ops.nf4_matmul(W, bf16_to_dev(d["x"]))
    dX = ops.nf4_matmul(W, bf16_to_dev(d["dY"]), transpose_w=True, out_f32=True)
    torch.cuda.synchronize()
    zA = np.zeros_like(d["A"])
    zB = np.zeros_like(d["B"])
    yo, _ = orc.lora_fwd(d["x"], Wq, zA, zB, None, 0.0)
    dXo, _, _ = orc.lora_bwd(d["x"], Wq, zA, zB, None, d["dY"], 0.0)
    assert rel(to_f64(y), yo) <= TOL
    assert rel(to_f64(dX), dXo) <= 1e-4


@pytest.mark.parametrize("M,N,K", [(300, 896, 1088), (512, 3584, 3584)])
def test_outputs_only_16_byte_aligned(ops, orc, M, N, K):
    """Outputs whose rows start 16 (not 32) bytes into an allocation take the
    16-byte store path of the epilogues; they hold the same bits as outputs
    at 32-byte aligned addresses (y, the bf16 and fp32 input gradients, and
    the accumulating fp32 input gradient)."""
    d, W, key = _linear(ops, orc, M, N, K, f"al{M}x{N}", lin=1, layer=1, step=3)
    x, A, B, dY = bf16_to_dev(d["x"]), f32_to_dev(d["A"]), f32_to_dev(d["B"]), bf16_to_dev(d["dY"])

    def shifted(shape, dtype, elems16):
        n = int(np.prod(shape))
        buf = torch.empty(n + 64, dtype=dtype, device="cuda")
        assert buf.data_ptr() % 32 == 0
        return buf[elems16:elems16 + n].view(shape)

    y, U, mask = ops.lora_linear_fwd(W, x, A, B, key)
    y2 = shifted((M, N), torch.bfloat16, 8)
    ops.lora_linear_fwd(W, x, A, B, key, y=y2)
    dXb, _, _ = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY)
    dXb2 = shifted((M, K), torch.bfloat16, 8)
    ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX=dXb2)
    dXf, _, _ = ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX_f32=True)
    dXf2 = shifted((M, K), torch.float32, 4)
    ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX=dXf2)
    base = torch.randn(M, K, device="cuda")
    acc1 = base.clone()
    ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX=acc1, accumulate=True)
    acc2 = shifted((M, K), torch.float32, 4)
    acc2.copy_(base)
    ops.lora_linear_bwd(W, x, A, B, key, U, mask, dY, dX=acc2, accumulate=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert y2.data_ptr() % 32 == 16 and dXf2.data_ptr() % 32 == 16
    assert torch.equal(y, y2)
    assert torch.equal(dXb, dXb2)
    assert torch.equal(dXf, dXf2)
    assert torch.equal(acc1, acc2)
