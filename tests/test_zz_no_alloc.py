"""moe_align_permute_noalloc: the expert sort for callers that cannot allocate
device memory when they call (its scratch is a fixed array inside the library).

Both entry points are called through the C ABI on the same routed ids and every
output must be identical (the sort is integer work: bit-exact), and the
no-allocation sort must equal the oracle's stable sort of the same ids.  Two calls
in a row, of different sizes, check that what the shared array keeps from the
first call does not leak into the second.  This file is collected last so that a run
stopping at the first failure has run everything else first.
"""
import ctypes

import pytest
import torch

import block_fp8_mixture_topk_gb300 as moe
from block_fp8_mixture_topk_gb300 import ops
from moe_testutil import check_sort

pytestmark = pytest.mark.gpu
DEV = "cuda"
MOE_ERR_WORKSPACE_TOO_SMALL = -3
SCRATCH_INTS = 262144          # MOE_NOALLOC_SORT_SCRATCH_INTS


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def sort_noalloc(ids, E, block_m=128):
    """Outputs of moe_align_permute_noalloc, laid out like the binding's moe_align_permute."""
    T, k = ids.shape
    rows = moe.moe_max_padded_rows(T, k, E, block_m)
    tiles = moe.moe_max_tiles(T, k, E, block_m)
    i32 = dict(dtype=torch.int32, device=ids.device)
    out = dict(expert_offsets=torch.empty(E + 1, **i32), padded_offsets=torch.empty(E + 1, **i32),
               sorted_pair_ids=torch.full((max(rows, 1),), -1, **i32), pos=torch.empty(max(T * k, 1), **i32),
               tile_expert=torch.empty(max(tiles, 1), **i32), tile_row0=torch.empty(max(tiles, 1), **i32),
               num_tiles=torch.empty(1, **i32))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = ops.lib().moe_align_permute_noalloc(_p(ids), T, k, E, block_m, _p(out["expert_offsets"]),
                                             _p(out["padded_offsets"]), _p(out["sorted_pair_ids"]), _p(out["pos"]),
                                             _p(out["tile_expert"]), _p(out["tile_row0"]), _p(out["num_tiles"]),
                                             stream)
    assert rc == 0, rc
    return out


def assert_same_sort(a, b, T, k):
    n = int(a["num_tiles"].item())
    used = int(a["padded_offsets"][-1].item())
    assert int(b["num_tiles"].item()) == n
    for key in ("expert_offsets", "padded_offsets"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["sorted_pair_ids"][:used], b["sorted_pair_ids"][:used])
    assert torch.equal(a["pos"][:T * k], b["pos"][:T * k])
    assert torch.equal(a["tile_expert"][:n], b["tile_expert"][:n])
    assert torch.equal(a["tile_row0"][:n], b["tile_row0"][:n])


def routed_ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ids[: T // 3, 0] = 1                      # one heavily loaded expert: several tiles
    return ids.to(DEV)


def test_noalloc_sort_matches_workspace_sort_on_two_calls_in_a_row():
    moe.moe_get_device_status(clear=True)
    cases = [(4096, 8, 256, 11), (300, 2, 8, 12)]   # a large problem, then a small one
    for T, k, E, seed in cases:
        ids = routed_ids(T, k, E, seed)
        want = moe.moe_align_permute(ids, E)
        got = sort_noalloc(ids, E)
        torch.cuda.synchronize()
        assert_same_sort(want, got, T, k)
        check_sort(got, ids.cpu().numpy(), E)
    assert moe.moe_get_device_status(clear=True) == 0


@pytest.mark.parametrize("T,k,E,block_m", [
    (8192, 32, 1024, 128),    # 256 chunks x 1024 experts: exactly the whole scratch
    (3000, 4, 1024, 64),      # the largest expert count, 64-row tiles
    (5000, 6, 64, 1),         # one-row "tiles"
    (700, 3, 96, 1000),       # tiles of 1000 rows
])
def test_noalloc_sort_equals_the_oracle(T, k, E, block_m):
    """Expert counts up to the library's maximum (1024) and tile sizes other than 128, against the
    oracle's stable sort, bit for bit."""
    moe.moe_get_device_status(clear=True)
    assert -(-T * k // 1024) * E <= SCRATCH_INTS
    ids = routed_ids(T, k, E, T + E + block_m)
    got = sort_noalloc(ids, E, block_m)
    torch.cuda.synchronize()
    check_sort(got, ids.cpu().numpy(), E, block_m)
    assert moe.moe_get_device_status(clear=True) == 0


def test_noalloc_sort_rejects_problems_beyond_its_scratch():
    E = 1024
    T = (SCRATCH_INTS // E + 1) * 1024          # one chunk of 1024 pairs too many, top-1
    p = ctypes.c_void_p(0x1000)
    rc = ops.lib().moe_align_permute_noalloc(p, T, 1, E, 128, p, p, p, p, p, p, p, None)
    assert rc == MOE_ERR_WORKSPACE_TOO_SMALL
