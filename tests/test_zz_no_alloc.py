"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device memory.

Such callers (code under a runtime that owns every device allocation, or that must
not call cudaMalloc at that point) cannot hand the library a workspace, so this
entry point keeps its scratch in a fixed 4 MiB array inside the library. This file
checks, through the C ABI, that two calls in a row give exactly what moe_dispatch
gives with a caller workspace, and exactly what the CPU oracle's stable counting
sort gives (integer and copy results, so bit-exact, which is the bound the dispatch
tests use), and that shapes beyond the fixed scratch are refused.
It is collected last so that a failure here comes after every other test has run.
"""
import ctypes

import pytest
import torch

import oracle
import workloads
from gpu_cases import check_dispatch_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    assert torch.cuda.is_available()
    return m


def _same_as_dispatch(moe, T, d, E, k, seed):
    wl = workloads.Workload("noalloc", T=T, d=d, E=E, k=k, f=64, seed=seed, backward=False)
    inp = workloads.make_inputs(wl)
    s = moe.shape(T, d, E, k, 64)
    x = inp.x.cuda()
    ids, _ = moe.route(inp.logits.cuda(), k)
    want = moe.dispatch(s, x, ids)
    got = moe.dispatch_noalloc(s, x, ids)
    torch.cuda.synchronize()
    P = int(want["padded_offsets"][-1])
    for key in ("counts", "offsets", "padded_offsets", "row_of", "tok_of"):
        assert torch.equal(got[key], want[key]), key
    assert torch.equal(got["xp"][:P], want["xp"][:P])
    # and against the oracle directly: counts, offsets, permutation and row copies
    rid, _ = oracle.route(inp.logits.numpy(), k)
    ref = oracle.dispatch(rid, E)
    ref["ids"] = rid
    check_dispatch_exact(got, ref, inp.x, k)


def test_two_calls_in_a_row_match_the_workspace_dispatch(moe):
    # the second call has a different shape, so it runs over the first call's leftovers
    _same_as_dispatch(moe, 4096, 2048, 128, 8, seed=71)
    _same_as_dispatch(moe, 65536, 64, 32, 4, seed=72)


def test_shapes_beyond_the_fixed_scratch_are_refused(moe):
    s = moe.shape(1 << 18, 64, 32, 8, 64)          # 2^21 assignments > 2^20 scratch entries
    p = ctypes.c_void_p(1 << 20)
    rc = moe.lib().moe_dispatch_noalloc(s, p, p, p, p, p, p, p, p, None)
    assert rc == -4                                 # MOE_ERR_WORKSPACE
