"""GPU parity of the grouped per-linear calls (ws_lora_linear_fwd_group /
_bwd_group) against the CPU oracle: several NF4-LoRA linears that read the
same input, as a layer's q, k, v (forward) or gate and up (both directions)
do.  Per linear: dropout bits bit-exact, y and the gradients within TOL of
the fp64 oracle, U within 1e-5; the grouped backward's fp32 input gradient
is the sum over the linears (within 1e-4 of the oracle's sum).  A repeated
call gives the same bits.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_to_dev, f32_to_dev, rel, to_f64

pytestmark = pytest.mark.gpu

P = 0.1
S = 2.0 / (1.0 - P)


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _group(ops, orc, M, Ns, K, tag, seed=3):
    from weight_streaming_nf4_gb300 import synth
    x = synth.normal_bf16(seed, f"{tag}.x", (M, K), 1.0)
    lins = []
    for g, N in enumerate(Ns):
        d = synth.linear_inputs(seed, M, N, K, 16, tag=f"{tag}.{g}")
        codes, absmax = ops.quantize_nf4(bf16_to_dev(d["W"]))
        Wq = orc.dequant_nf4(*orc.quantize_nf4(d["W"]))
        key = ops.dropout_key(seed=seed, step=2, layer=1, linear=g, p=P)
        lins.append(dict(d=d, W=ops.NF4Weight(codes, absmax, N, K), Wq=Wq, key=key,
                         om=orc.dropout_mask(seed, 2, 1, g, 0, P, M, K)))
    return x, lins


@pytest.mark.parametrize("M,Ns,K", [
    (512, (512, 128, 128), 512),     # q, k, v of a small layer: one grouped GEMM (widths % 128 == 0)
    (300, (896, 128, 128), 896),     # 0.5B q, k, v widths, ragged M
    (200, (4864, 4864), 896),        # 0.5B gate, up
])
def test_group_forward(ops, orc, M, Ns, K):
    xb, lins = _group(ops, orc, M, Ns, K, f"gf{M}{K}")
    x = bf16_to_dev(xb)
    Ws = [l["W"] for l in lins]
    As = [f32_to_dev(l["d"]["A"]) for l in lins]
    Bs = [f32_to_dev(l["d"]["B"]) for l in lins]
    keys = [l["key"] for l in lins]
    ys, Us, masks = ops.lora_linear_fwd_group(Ws, x, As, Bs, keys)
    ys2, Us2, masks2 = ops.lora_linear_fwd_group(Ws, x, As, Bs, keys)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    for g, l in enumerate(lins):
        assert np.array_equal(masks[g].cpu().numpy().view(np.uint32), l["om"]), g
        yo, Uo = orc.lora_fwd(xb, l["Wq"], l["d"]["A"], l["d"]["B"], l["om"], S)
        assert rel(to_f64(ys[g]), yo) <= TOL, g
        assert rel(to_f64(Us[g]), Uo) <= 1e-5, g
        assert torch.equal(ys[g], ys2[g]) and torch.equal(Us[g], Us2[g])


@pytest.mark.parametrize("M,N,K,ng", [(200, 4864, 896, 2), (512, 128, 896, 2), (256, 512, 512, 3)])
def test_group_backward(ops, orc, M, N, K, ng):
    xb, lins = _group(ops, orc, M, (N,) * ng, K, f"gb{M}{N}{K}")
    x = bf16_to_dev(xb)
    Ws = [l["W"] for l in lins]
    As = [f32_to_dev(l["d"]["A"]) for l in lins]
    Bs = [f32_to_dev(l["d"]["B"]) for l in lins]
    keys = [l["key"] for l in lins]
    dYs = [bf16_to_dev(l["d"]["dY"]) for l in lins]
    _, Us, masks = ops.lora_linear_fwd_group(Ws, x, As, Bs, keys)
    dX, dAs, dBs = ops.lora_linear_bwd_group(Ws, x, As, Bs, keys, Us, masks, dYs)
    dX2, dAs2, dBs2 = ops.lora_linear_bwd_group(Ws, x, As, Bs, keys, Us, None, dYs)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    dX_ref = np.zeros((M, K))
    for g, l in enumerate(lins):
        dXo, dAo, dBo = orc.lora_bwd(xb, l["Wq"], l["d"]["A"], l["d"]["B"], l["om"], l["d"]["dY"], S)
        dX_ref += dXo
        assert rel(to_f64(dAs[g]), dAo) <= TOL, g
        assert rel(to_f64(dBs[g]), dBo) <= TOL, g
        # masks regenerated from the keys give the same gradients
        assert torch.equal(dAs[g], dAs2[g]) and torch.equal(dBs[g], dBs2[g])
    assert rel(to_f64(dX), dX_ref) <= 1e-4
    assert torch.equal(dX, dX2)


def test_group_rejects_bf16_sum(ops, orc):
    xb, lins = _group(ops, orc, 64, (128, 128), 256, "rej")
    x = bf16_to_dev(xb)
    Ws = [l["W"] for l in lins]
    As = [f32_to_dev(l["d"]["A"]) for l in lins]
    Bs = [f32_to_dev(l["d"]["B"]) for l in lins]
    keys = [l["key"] for l in lins]
    _, Us, masks = ops.lora_linear_fwd_group(Ws, x, As, Bs, keys)
    dX = torch.empty((64, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.WsError):
        ops.lora_linear_bwd_group(Ws, x, As, Bs, keys, Us, masks,
                                  [bf16_to_dev(l["d"]["dY"]) for l in lins], dX=dX)
