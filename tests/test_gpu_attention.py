"""GPU parity of the causal attention core (ws_attention_fwd / _bwd) against
the fp64 oracle.

The core is scaled dot-product attention, causal, with grouped kv heads
(query head h reads kv head h // (nh / nkv)); the research page "Poros"
keeps the model's own attention under streaming.  Inputs are bf16 draws of
N(0, sigma^2): sigma = 1 gives a spread-out softmax, sigma = 3 a peaked one
(scores with a standard deviation near 9).  Shapes cover the 32B layer
(40 query heads over 8 kv heads, head_dim 128, 512 tokens), the 0.5B
layer's grouping (14 over 2, head_dim 64), several sequences per launch,
ragged lengths (1, 130, 200 tokens: partial 64- and 128-row tiles and tiles
that straddle two sequences).

Checks:
- the fp32 output o32 within 1e-4 normwise of the oracle (the probabilities
  enter the products as two bf16 parts), the bf16 output the bf16 rounding
  of o32 bit for bit, the log-sum-exp within 1e-5 relative;
- dq, dk, dv (bf16) within TOL normwise of the oracle's gradients computed
  from the same bf16 dO, and elementwise within one bf16 ulp of the oracle
  plus 1e-3 of the tensor's rms;
- the same call twice gives the same bits, and a sequence of a batch gives
  the same bits as that sequence alone.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_bits, bf16_to_dev, rel, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _inputs(seed, M, nh, nkv, d, sigma):
    from weight_streaming_nf4_gb300 import synth
    q = synth.normal_bf16(seed, "attn.q", (M, nh * d), sigma)
    k = synth.normal_bf16(seed, "attn.k", (M, nkv * d), sigma)
    v = synth.normal_bf16(seed, "attn.v", (M, nkv * d), 1.0)
    dO = synth.normal_bf16(seed, "attn.dO", (M, nh * d), 1.0)
    return q, k, v, dO


def _f64(bits):
    from weight_streaming_nf4_gb300 import synth
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _ulp_check(gpu, ref):
    """Elementwise: |gpu - ref| <= 2^-8 |ref| + 1e-3 rms(ref) + 1e-5.  The
    absolute 1e-5 (inputs are O(1)) covers gradients that vanish exactly,
    e.g. dq and dk of a one-token sequence, where fp32 rounding of
    dO.v - dO.o leaves about 1e-7."""
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bad = np.abs(gpu - ref) > 2.0 ** -8 * np.abs(ref) + 1e-3 * rms + 1e-5
    assert not bad.any(), (int(bad.sum()), float(np.max(np.abs(gpu - ref))))


CASES = [
    # n_seq, S, nh, nkv, d, sigma
    (1, 512, 40, 8, 128, 1.0),    # the 32B layer's attention
    (1, 512, 8, 2, 128, 3.0),     # peaked softmax
    (2, 200, 14, 2, 64, 1.0),     # 0.5B grouping, two ragged sequences
    (1, 130, 5, 1, 128, 1.0),     # ragged tail of 2 tokens
    (3, 1, 4, 2, 64, 1.0),        # one token per sequence
    (4, 96, 4, 4, 128, 2.0),      # no grouping, sequences inside one tile
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}_s{c[1]}_h{c[2]}_kv{c[3]}_d{c[4]}_sig{c[5]}"
                                             for c in CASES])
def test_attention_parity(ops, orc, case):
    n_seq, S, nh, nkv, d, sigma = case
    M = n_seq * S
    qb, kb, vb, dOb = _inputs(7, M, nh, nkv, d, sigma)
    q, k, v, dO = (bf16_to_dev(a) for a in (qb, kb, vb, dOb))
    o, o32, lse = ops.attention_fwd(q, k, v, n_seq, d)
    dq, dk, dv = ops.attention_bwd(q, k, v, o32, lse, dO, n_seq, d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0

    q64, k64, v64, dO64 = _f64(qb), _f64(kb), _f64(vb), _f64(dOb)
    o_ref, lse_ref = orc.attention_fwd(q64, k64, v64, n_seq, d, want_lse=True)
    assert rel(to_f64(o32), o_ref) <= 1e-4
    o32_np = o32.cpu().numpy()
    from weight_streaming_nf4_gb300 import synth
    np.testing.assert_array_equal(bf16_bits(o), synth.to_bf16_bits(o32_np))
    np.testing.assert_allclose(lse.cpu().numpy().astype(np.float64), lse_ref, rtol=1e-5, atol=1e-5)

    dq_ref, dk_ref, dv_ref = orc.attention_bwd(q64, k64, v64, dO64, n_seq, d)
    for name, g, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        e = rel(to_f64(g), ref)
        assert e <= TOL, (name, e)
        _ulp_check(to_f64(g), ref)


def test_attention_repeats_bitwise_and_batches_split(ops):
    n_seq, S, nh, nkv, d = 2, 300, 8, 2, 128
    M = n_seq * S
    qb, kb, vb, dOb = _inputs(11, M, nh, nkv, d, 1.5)
    q, k, v, dO = (bf16_to_dev(a) for a in (qb, kb, vb, dOb))
    r1 = ops.attention_fwd(q, k, v, n_seq, d)
    g1 = ops.attention_bwd(q, k, v, r1[1], r1[2], dO, n_seq, d)
    r2 = ops.attention_fwd(q, k, v, n_seq, d)
    g2 = ops.attention_bwd(q, k, v, r2[1], r2[2], dO, n_seq, d)
    for a, b in zip(list(r1) + list(g1), list(r2) + list(g2)):
        assert torch.equal(a, b)
    # the second sequence on its own
    sl = slice(S, 2 * S)
    q2, k2, v2, dO2 = (t[sl].contiguous() for t in (q, k, v, dO))
    s_o, s_o32, s_lse = ops.attention_fwd(q2, k2, v2, 1, d)
    s_dq, s_dk, s_dv = ops.attention_bwd(q2, k2, v2, s_o32, s_lse, dO2, 1, d)
    torch.cuda.synchronize()
    assert torch.equal(s_o, r1[0][sl]) and torch.equal(s_o32, r1[1][sl])
    assert torch.equal(s_lse, r1[2][:, sl])
    assert torch.equal(s_dq, g1[0][sl]) and torch.equal(s_dk, g1[1][sl])
    assert torch.equal(s_dv, g1[2][sl])
    assert ops.device_error() == 0


def test_attention_outputs_only_16_byte_aligned(ops):
    """O, the fp32 O, dQ and the backward workspace (the per-head dK/dV
    partials) starting 16 bytes into 32-byte aligned allocations take the
    16-byte store path; the results hold the same bits."""
    g = torch.Generator().manual_seed(5)
    S, nh, nkv, d = 256, 8, 2, 128
    q = (torch.randn(S, nh * d, generator=g)).to(torch.bfloat16).cuda()
    k = (torch.randn(S, nkv * d, generator=g)).to(torch.bfloat16).cuda()
    v = (torch.randn(S, nkv * d, generator=g)).to(torch.bfloat16).cuda()
    dO = (torch.randn(S, nh * d, generator=g)).to(torch.bfloat16).cuda()

    def shifted(shape, dtype, elems16):
        n = int(np.prod(shape))
        buf = torch.empty(n + 64, dtype=dtype, device="cuda")
        assert buf.data_ptr() % 32 == 0
        return buf[elems16:elems16 + n].view(shape)

    o, o32, lse = ops.attention_fwd(q, k, v, 1, d)
    o2 = shifted((S, nh * d), torch.bfloat16, 8)
    o32b = shifted((S, nh * d), torch.float32, 4)
    ops.attention_fwd(q, k, v, 1, d, o=o2, o32=o32b)
    dq, dk, dv = ops.attention_bwd(q, k, v, o32, lse, dO, 1, d)
    wsz = ops.attention_workspace_size(S, nh, d)
    ws = torch.empty(wsz + 64, dtype=torch.uint8, device="cuda")[16:16 + wsz]
    dq2 = shifted((S, nh * d), torch.bfloat16, 8)
    _, dk2, dv2 = ops.attention_bwd(q, k, v, o32, lse, dO, 1, d, dq=dq2, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert o2.data_ptr() % 32 == 16 and ws.data_ptr() % 32 == 16
    assert torch.equal(o, o2) and torch.equal(o32, o32b)
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_attention_rejects_bad_arguments(ops):
    q = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.WsError):
        ops.attention_fwd(q, k, k, 1, 32)            # head_dim 32 unsupported
    with pytest.raises(ops.WsError):
        ops.attention_fwd(q[:, 1:], k, k, 1, 64)     # misaligned rows
