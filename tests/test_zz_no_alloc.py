"""The allocation-free dispatch entry point against the workspace version.

moe_build_dispatch_noalloc serves callers that cannot allocate device memory
(hosts that own all device memory, or loops where an allocation's implicit
synchronisation is not acceptable): its scratch is a static device array in the
library. It must give exactly the same index as moe_build_dispatch, call after
call, since the array keeps the previous call's contents, and after its first
call on a device (which may load the library's device code and the array) it
must leave the device's free memory unchanged. This file is named to be
collected last."""
import pytest
import torch

from token_dispatch_grouped_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run_both(B, T, E, K, ids):
    s = B.shape(T, 128, E, K, 128)
    TK = T * K
    dev = "cuda"
    ws = torch.empty(B.moe_workspace_size(s, B.MOE_WS_DISPATCH), dtype=torch.uint8, device=dev)
    ref = [torch.full((TK,), -7, dtype=torch.int32, device=dev),
           torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
           torch.full((TK,), -7, dtype=torch.int32, device=dev)]
    out = [torch.full_like(t, -9) for t in ref]
    B.moe_build_dispatch(s, ids, *ref, ws)
    B.moe_build_dispatch_noalloc(s, ids, *out)
    assert B.moe_get_error() == B.MOE_OK
    return ref, out


def test_noalloc_dispatch_matches_workspace_version_two_calls():
    from token_dispatch_grouped_gb300 import binding as B
    cases = [(3000, 64, 6, I.random_ids(3000, 64, 6, seed=11, skew=1.1)),
             (513, 16, 4, I.random_ids(513, 16, 4, seed=12))]
    for T, E, K, ids in cases:                       # two calls in a row, different shapes
        ref, out = _run_both(B, T, E, K, ids.cuda())
        for a, b in zip(ref, out):
            assert torch.equal(a, b)
    # the same shape again: the array still holds the previous call's data
    T, E, K, ids = cases[0]
    ref, out = _run_both(B, T, E, K, ids.cuda())
    for a, b in zip(ref, out):
        assert torch.equal(a, b)


def test_noalloc_dispatch_rejects_shapes_beyond_static_limit():
    from token_dispatch_grouped_gb300 import binding as B
    T, E, K = 256 * 4097, 256, 2                      # 4097 blocks x 256 experts > 2^20 entries
    s = B.shape(T, 128, E, K, 128)
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    rc = B.moe_build_dispatch_noalloc(s, dummy, dummy, dummy, dummy, check=False)
    assert rc == B.MOE_ERR_STATIC_SCRATCH_LIMIT


def test_noalloc_dispatch_changes_no_device_memory():
    from token_dispatch_grouped_gb300 import binding as B
    T, E, K = 4000, 32, 4
    s = B.shape(T, 128, E, K, 128)
    ids = I.random_ids(T, E, K, seed=13).cuda()
    eti = torch.empty(T * K, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    tim = torch.empty(T * K, dtype=torch.int32, device="cuda")
    B.moe_build_dispatch_noalloc(s, ids, eti, off, tim)   # first call: set-up, module load
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    torch_alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        B.moe_build_dispatch_noalloc(s, ids, eti, off, tim)
    torch.cuda.synchronize()
    assert B.moe_get_error() == B.MOE_OK
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == torch_alloc0
