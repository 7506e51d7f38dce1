"""ws_nf4_matmul_noalloc: the frozen NF4 product for callers that cannot
allocate device memory (a framework that owns the allocator, a plugin without
allocation hooks, a path that must not allocate once running).  Its split
partials live in the library's built-in device scratch array instead of a
caller workspace.  Checked through the C ABI against ws_nf4_matmul, which
takes a caller workspace: both run the same plan and kernel on the same
inputs, so the outputs must be identical bit for bit, on two calls in a row
per shape (the second call reuses scratch the first one left behind), in
bf16 and fp32 output, on the default stream and on a created one.  Collected
last so a failure here does not stop the rest of a stop-at-first-failure run.
"""
import pytest
import torch

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


@pytest.mark.parametrize("M,N,K,tw,f32", [(512, 5120, 5120, False, True),
                                           (512, 5120, 5120, True, False),
                                           (64, 512, 4096, False, False),
                                           (300, 896, 1088, True, True),
                                           (512, 27648, 5120, False, False)])
@pytest.mark.parametrize("own_stream", [False, True])
def test_noalloc_matches_workspace_version(ops, M, N, K, tw, f32, own_stream):
    W, g = _weight(ops, N, K, M + N + K)
    act = torch.randn(M, N if tw else K, generator=g, device="cuda:0").to(torch.bfloat16)
    ref = ops.nf4_matmul(W, act, transpose_w=tw, out_f32=f32)
    out = torch.empty_like(ref)
    st = torch.cuda.Stream() if own_stream else torch.cuda.current_stream()
    st.wait_stream(torch.cuda.current_stream())
    for _ in range(2):
        with torch.cuda.stream(st):
            out.fill_(float("nan"))
            ops.nf4_matmul_noalloc(W, act, transpose_w=tw, out=out, stream=st)
        st.synchronize()
        assert torch.equal(out, ref)
    assert ops.device_error() == 0


def test_noalloc_uses_scratch_and_every_plan_fits(ops):
    # a shape that splits its contraction really goes through the scratch array
    assert ops.nf4_matmul_workspace_size(512, 5120, 5120) > 256
    # the split partials are at most one 256 x 256 fp32 tile per resident CTA,
    # so on this GPU every shape fits the built-in array and WS_ERR_OOM (the
    # check that precedes every launch) cannot occur: the largest plans here
    for M, N, K, tw in [(512, 27648, 5120, False), (4096, 65536, 8192, False),
                        (4096, 8192, 29568, True), (1 << 16, 1 << 16, 8192, False)]:
        assert ops.nf4_matmul_workspace_size(M, N, K, tw) <= ops.NOALLOC_SCRATCH_BYTES
