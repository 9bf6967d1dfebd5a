"""lmoe_segments_noalloc: the entry point for callers that cannot let the library
allocate device memory (their memory belongs to another allocator, or cudaMalloc's
implicit synchronisation is not acceptable on their path).  It must produce exactly the
segments the allocating entry point (lmoe_route) leaves in its workspace, on consecutive
calls that reuse its fixed scratch array.  Collected last so a failure here comes after
every other test has run."""
import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O
from sparse_moe_layer_cutoff_b300 import LatentMoE
from sparse_moe_layer_cutoff_b300 import lmoe as L
from sparse_moe_layer_cutoff_b300.lmoe import workspace_tensors
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _reference_segments(w, bt):
    """Segments from the existing entry point: lmoe_route on a context with a workspace."""
    x, weights, bias = make_inputs(w, "cuda", bt)
    layer = LatentMoE(w.shape, weights, max_bt=bt, router_bias=bias)
    r = layer.route(x)
    torch.cuda.synchronize()
    ws = workspace_tensors(layer)
    ref = {k: ws[k].clone() for k in ("offsets", "perm", "inv")}
    ref["counts"] = r["counts"].clone()
    ref["idx"] = r["idx"].clone()
    layer.close()
    return ref


def _noalloc(idx, n_experts):
    bt, K = idx.shape
    out = dict(counts=torch.full((n_experts,), -1, dtype=torch.int32, device="cuda"),
               offsets=torch.full((n_experts + 1,), -1, dtype=torch.int32, device="cuda"),
               perm=torch.full((bt * K,), -1, dtype=torch.int32, device="cuda"),
               inv=torch.full((bt, K), -1, dtype=torch.int32, device="cuda"))
    st = L.lmoe_segments_noalloc(idx.data_ptr(), bt, K, n_experts, out["counts"].data_ptr(),
                                 out["offsets"].data_ptr(), out["perm"].data_ptr(), out["inv"].data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == L.LMOE_OK, L.lmoe_status_string(st)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,bt", [("small_bf16", 2048), ("full_decode_bt64", 64)])
def test_noalloc_segments_match_allocating_entry_point(name, bt):
    w = WORKLOADS[name]
    ref = _reference_segments(w, bt)
    E = w.shape.n_experts
    # two calls in a row (the second reuses what the first left in the scratch array),
    # then a call of another size, then the first size again
    first = _noalloc(ref["idx"], E)
    second = _noalloc(ref["idx"], E)
    small = _noalloc(ref["idx"][: max(1, bt // 3)].contiguous(), E)
    third = _noalloc(ref["idx"], E)
    for got in (first, second, third):
        for k in ("counts", "offsets", "perm", "inv"):
            assert torch.equal(got[k], ref[k]), k           # integer outputs: bit-exact
    # every call, the smaller one after a larger one included (stale per-block counts in the
    # shared scratch would show there), against the oracle's stable counting sort
    for got, ids in ((first, ref["idx"]), (small, ref["idx"][: max(1, bt // 3)]), (third, ref["idx"])):
        idx = ids.cpu().numpy()
        off, perm, inv = O.permutation(idx, E)
        np.testing.assert_array_equal(got["counts"].cpu().numpy(), O.expert_counts(idx, E))
        np.testing.assert_array_equal(got["offsets"].cpu().numpy(), off)
        np.testing.assert_array_equal(got["perm"].cpu().numpy(), perm)
        np.testing.assert_array_equal(got["inv"].cpu().numpy(), inv)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    idx = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    o = torch.zeros(8, dtype=torch.int32, device="cuda")
    # (ceil(bt/128) * E + 2E + 1) * 4 bytes > 4 MiB
    st = L.lmoe_segments_noalloc(idx.data_ptr(), 2_000_000, 2, 4096, o.data_ptr(), o.data_ptr(), o.data_ptr(),
                                 o.data_ptr(), 0)
    assert st == L.LMOE_ERR_UNSUPPORTED
    assert L.lmoe_segments_noalloc(0, 4, 2, 8, o.data_ptr(), o.data_ptr(), o.data_ptr(), o.data_ptr(), 0) \
        == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_segments_noalloc(idx.data_ptr(), 0, 2, 8, o.data_ptr(), o.data_ptr(), o.data_ptr(),
                                   o.data_ptr(), 0) == L.LMOE_OK
