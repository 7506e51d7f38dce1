"""The streamed NF4 loader (ws_stack_put_weight): the stack image is
built one tensor at a time, straight into HBM or through a one-tensor device
staging buffer into pinned host memory, so the GPU never holds more than one
bf16 weight and its NF4 form (research page "Poros", block-streamed NF4 loader
paragraphs).  The pages gate the loader on byte identity with a standard load;
here both images must equal, byte for byte, the image assembled from the
oracle's codes and block scales at the layout's offsets.
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_streaming_nf4_gb300 import ops as o
    return o


def _weights(cfg, seed):
    from weight_streaming_nf4_gb300 import synth
    names = ("q", "k", "v", "o", "gate", "up", "down")
    return {(layer, lin): synth.stack_weights(seed, layer, names[lin], N, K)[0]
            for layer in range(cfg.n_layers) for lin, (N, K) in enumerate(cfg.shapes())}


def _oracle_image(ops, orc, cfg, bl, W):
    sz = ops.stack_sizes(cfg, bl)
    bb = sz["block_bytes"]
    img = np.zeros(cfg.n_layers // bl * bb, np.uint8)
    for (layer, lin), w in W.items():
        codes, absmax = orc.quantize_nf4(w)
        oc, oa = ops.stack_weight_offset(cfg, layer % bl, lin)
        base = (layer // bl) * bb
        img[base + oc:base + oc + codes.size] = codes.ravel()
        a = absmax.view(np.uint8).ravel()
        img[base + oa:base + oa + a.size] = a
    return img


def test_loader_images_are_byte_identical_to_the_oracle(ops, orc):
    cfg = ops.StackCfg(M=64, H=896, KV=128, I=4864, head_dim=64, n_layers=4)
    bl = 2
    W = _weights(cfg, 11)
    ref = _oracle_image(ops, orc, cfg, bl, W)
    n = ref.size
    host = torch.zeros(n, dtype=torch.uint8, pin_memory=True)
    devimg = torch.zeros(n, dtype=torch.uint8, device="cuda:0")
    staging = torch.empty(ops.stack_loader_staging_bytes(cfg), dtype=torch.uint8, device="cuda:0")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    largest = 0
    for (layer, lin), w in W.items():
        Wd = bf16_to_dev(w)
        largest = max(largest, Wd.numel() * 2)
        ops.stack_put_weight(cfg, bl, layer, lin, Wd, host, staging)
        ops.stack_put_weight(cfg, bl, layer, lin, Wd, devimg)
        del Wd
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    # the GPU held one bf16 tensor at a time (plus the images and staging allocated before)
    assert torch.cuda.max_memory_allocated() - base <= largest + (2 << 20)
    assert np.array_equal(host.numpy(), ref)
    assert np.array_equal(devimg.cpu().numpy(), ref)


def test_loader_argument_errors(ops):
    cfg = ops.StackCfg(M=64, H=256, KV=64, I=512, head_dim=32, n_layers=2)
    n = 2 * ops.stack_sizes(cfg, 1)["block_bytes"]
    host = torch.zeros(n, dtype=torch.uint8, pin_memory=True)
    staging = torch.empty(ops.stack_loader_staging_bytes(cfg), dtype=torch.uint8, device="cuda:0")
    W = torch.zeros(512, 256, dtype=torch.bfloat16, device="cuda:0")  # gate's shape
    with pytest.raises(ops.WsError) as e:
        ops.stack_put_weight(cfg, 1, 0, 0, W, host, staging)     # q is [256, 256]
    assert e.value.status == -2
    with pytest.raises(ops.WsError) as e:
        ops.stack_put_weight(cfg, 1, 0, 4, W, host, staging[:1024])
    assert e.value.status == -6
    with pytest.raises(ops.WsError) as e:
        ops.stack_put_weight(cfg, 1, 2, 4, W, host, staging)     # layer out of range
    assert e.value.status == -1
    pageable = torch.zeros(n, dtype=torch.uint8)
    with pytest.raises(ops.WsError) as e:
        ops.stack_put_weight(cfg, 1, 0, 4, W, pageable, staging)
    assert e.value.status == -8
