"""The allocation-free route map agrees with the workspace version and with
the oracle.

moe_expert_offsets_noalloc serves callers that cannot allocate device memory
(stream capture, engines that hand over only their own arena's tensors,
real-time loops): its scratch is a static device array inside libmoe instead
of a caller workspace.  It must give exactly the outputs of moe_expert_offsets
(integer outputs: bit-exact), call after call, since every call reuses the
same array.  This file sorts last so a stop-at-first-failure run has already
run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np

import oracle.layer as ol
import pytest
import torch

from token_dispatch_grouped_router_gb300 import libmoe as L

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_inputs(T, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[idx == 1] = 2                       # leave expert 1 empty
    return torch.from_numpy(idx).to(DEV)


def _outputs(T, k, E):
    i32 = torch.int32
    return (torch.full((E,), -7, dtype=i32, device=DEV), torch.full((E + 1,), -7, dtype=i32, device=DEV),
            torch.full((T * k,), -7, dtype=i32, device=DEV), torch.full((T * k,), -7, dtype=i32, device=DEV))


@pytest.mark.parametrize("T,k,E", [(16384, 4, 128), (1000, 2, 8), (65536, 4, 1024)])
def test_no_alloc_route_map_equals_workspace_route_map(T, k, E):
    ensure_built()
    L.load()
    ws = torch.zeros(L.moe_workspace_size(T, E, k, 64, 64), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(2):                  # two calls in a row share the static scratch
        idx = _route_inputs(T, k, E, seed=call)
        ref = _outputs(T, k, E)
        got = _outputs(T, k, E)
        L.moe_expert_offsets(idx, E, *ref, ws)
        L.moe_expert_offsets_noalloc(idx, E, *got, status)
        torch.cuda.synchronize()
        names = ("counts", "offsets", "row_of_slot", "slot_of_row")
        for a, b, name in zip(got, ref, names):
            assert torch.equal(a, b), (call, name)
        # bit-exact against the plain definition as well (expert 1 is empty)
        for a, o, name in zip(got, ol.route_map(idx.cpu().numpy(), E), names):
            assert np.array_equal(a.cpu().numpy(), o), (call, name, "oracle")
        assert int(status.item()) == 0
        assert L.moe_get_status(ws) == 0


def test_no_alloc_reports_bad_ids_and_rejects_oversize():
    ensure_built()
    lib = L.load()
    T, k, E = 64, 2, 8
    idx = _route_inputs(T, k, E, seed=3)
    idx[5, 1] = E + 1
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _outputs(T, k, E)
    L.moe_expert_offsets_noalloc(idx, E, *out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1          # MOE_DEV_BAD_EXPERT_ID
    # beyond the static scratch (T * k > 262144): a clear error, nothing launched
    before = L.moe_launch_count()
    fake = ctypes.c_void_p(out[0].data_ptr())
    rc = lib.moe_expert_offsets_noalloc(fake, 262145, 1, 8, fake, fake, fake, fake, None, None)
    assert rc == -2                          # MOE_ERR_UNSUPPORTED
    assert L.moe_launch_count() == before
    # the binding checks the optional status word like every other output
    for bad in (torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int64, device=DEV),
                torch.zeros(0, dtype=torch.int32, device=DEV)):
        with pytest.raises(ValueError):
            L.moe_expert_offsets_noalloc(idx, E, *out, bad)
    assert L.moe_launch_count() == before
