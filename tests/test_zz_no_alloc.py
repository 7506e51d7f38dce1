"""ws_nf4_matmul_noalloc: the frozen NF4 product for callers that cannot
allocate device memory (a framework that owns the allocator, a plugin without
allocation hooks, a path that must not allocate once running).  Its split
partials live in the library's built-in device scratch array instead of a
caller workspace.  Checked through the C ABI against ws_nf4_matmul, which
takes a caller workspace, on two calls in a row per shape (the second call
reuses scratch the first one left behind).  Collected last so a failure here
does not stop the rest of a stop-at-first-failure run.
"""
import pytest
import torch

from gpu_util import TOL, rel, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _weight(ops, N, K, seed):
    g = torch.Generator(device="cuda:0").manual_seed(seed)
    W = (torch.randn(N, K, generator=g, device="cuda:0") * 0.02).to(torch.bfloat16)
    codes, absmax = ops.quantize_nf4(W)
    return ops.NF4Weight(codes, absmax, N, K), g


@pytest.mark.parametrize("M,N,K,tw", [(512, 5120, 5120, False), (512, 5120, 5120, True),
                                       (64, 512, 4096, False), (300, 896, 1088, True),
                                       (512, 27648, 5120, False)])
def test_noalloc_matches_workspace_version(ops, M, N, K, tw):
    W, g = _weight(ops, N, K, M + N + K)
    act = torch.randn(M, N if tw else K, generator=g, device="cuda:0").to(torch.bfloat16)
    ref = ops.nf4_matmul(W, act, transpose_w=tw, out_f32=True)
    out = torch.empty_like(ref)
    for _ in range(2):
        out.fill_(float("nan"))
        ops.nf4_matmul_noalloc(W, act, transpose_w=tw, out=out)
        torch.cuda.synchronize()
        assert rel(to_f64(out), to_f64(ref)) <= TOL
    assert ops.device_error() == 0


def test_noalloc_uses_scratch_and_rejects_oversize(ops):
    # a shape that splits its contraction really goes through the scratch array
    assert ops.nf4_matmul_workspace_size(512, 5120, 5120) > 256
    # a shape whose partials exceed the built-in array is refused up front
    M, N, K = 512, 9216, 4096
    if ops.nf4_matmul_workspace_size(M, N, K) <= ops.NOALLOC_SCRATCH_BYTES:
        pytest.skip("no oversize shape for this SM count")
    W, g = _weight(ops, N, K, 7)
    act = torch.randn(M, K, generator=g, device="cuda:0").to(torch.bfloat16)
    out = torch.empty(M, N, device="cuda:0", dtype=torch.bfloat16)
    with pytest.raises(ops.WsError) as e:
        ops.nf4_matmul_noalloc(W, act, out=out)
    assert e.value.status == -6
