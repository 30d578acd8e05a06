"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device memory (GPU).

Such callers (a plugin that only receives its input and output buffers from a host framework, or
a server whose device memory is fixed at start-up) cannot keep a workspace, so this entry point
uses a fixed scratch array inside the library. Its results must equal moe_dispatch's exactly
(integer and byte outputs), on two calls in a row with different problems, so that nothing of
the previous call's scratch leaks into the next. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from harness import bits_of, config_of, to_device
from mixture_experts_layer_96_b300 import Workspace, moe_dispatch
from mixture_experts_layer_96_b300 import moe as M
from workloads import WORKLOADS, Generator, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


def _compare(shape):
    cfg = config_of(shape)
    g = Generator(shape)
    b = shape.dtype == "bf16"
    x = to_device(g.x(), b)
    idx = torch.from_numpy(g.topk_idx()).cuda()
    ws = Workspace(cfg)
    want = moe_dispatch(cfg, x, idx, ws=ws)
    ws.check()
    got = M.moe_dispatch_noalloc(cfg, x, idx)
    torch.cuda.synchronize()
    kept = int(want[1][-1].item())
    for name, a, w in zip(("counts", "offsets", "slot_of", "row_token"), got[:4], want[:4]):
        np.testing.assert_array_equal(bits_of(a), bits_of(w), err_msg=name)
    np.testing.assert_array_equal(bits_of(got[4])[:kept], bits_of(want[4])[:kept])
    return kept


def test_noalloc_dispatch_equals_dispatch_on_two_calls_in_a_row():
    # first call: 64 experts with capacity drops; second call: 256 experts, fewer units, no drop
    a = scaled(WORKLOADS["skewed_bf16"], T=3000, h=256)
    b = scaled(WORKLOADS["finegrained_bf16"], T=500, h=256)
    ka = _compare(a)
    kb = _compare(b)
    assert ka < 3000 * 2 and kb == 500 * 8
    _compare(a)  # and back: a smaller scratch footprint after a larger one


def test_noalloc_dispatch_rejects_problems_past_its_scratch():
    """A problem whose scratch does not fit the fixed array is refused before anything is enqueued.
    Every buffer passed is real device memory of the full size the call would use, so even a call
    that wrongly went ahead would stay inside its buffers."""
    T, h, E, K = 200_000, 64, 256, 8   # 1563 chunks x 256 experts x 8 B > 1 MiB
    cfg = M.make_config(T, h, E, K, 64)
    dev = "cuda"
    x = torch.zeros((T, h), dtype=torch.bfloat16, device=dev)
    idx = torch.zeros((T, K), dtype=torch.int32, device=dev)
    counts = torch.empty((E,), dtype=torch.int32, device=dev)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
    slot_of = torch.empty((T, K), dtype=torch.int32, device=dev)
    row_token = torch.empty((T * K,), dtype=torch.int32, device=dev)
    x_packed = torch.empty((T * K, h), dtype=torch.bfloat16, device=dev)
    lib = M.load_library()
    before = M.launch_count()
    code = lib.moe_dispatch_noalloc(ctypes.byref(cfg), x.data_ptr(), idx.data_ptr(), counts.data_ptr(),
                                    offsets.data_ptr(), slot_of.data_ptr(), row_token.data_ptr(),
                                    x_packed.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == M.MOE_ERR_UNSUPPORTED
    assert M.launch_count() == before   # nothing was launched
    with pytest.raises(M.MoEError, match="fixed scratch"):
        M.moe_dispatch_noalloc(cfg, x, idx, counts=counts, offsets=offsets, slot_of=slot_of, row_token=row_token,
                               x_packed=x_packed)
