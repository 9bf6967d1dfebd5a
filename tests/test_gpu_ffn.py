"""Parity of the dense SiTU-GLU FFN (lmoe_ffn_*) with the fp64 oracle (GPU): outputs within
max-abs 2e-2 and relative L2 1e-2, the bf16 bound of the layer."""
import numpy as np
import pytest
import torch

from oracle import lmoe_oracle as O
from sparse_moe_layer_cutoff_b300 import DenseFFN, LmoeError
from sparse_moe_layer_cutoff_b300 import lmoe as L
from tests.lmoe_testing import BF16_MAX_ABS, BF16_REL_L2, rel_l2, to64
from workloads import FFN_WORKLOADS, make_ffn_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _oracle_rows(x, wg, wu, wd, w, rows, chunk=4096):
    """Oracle output for the given rows; the intermediate units are taken in chunks (the
    FFN is a sum over them) so that fp64 copies of large weights stay small."""
    xr = to64(x[rows])
    out = np.zeros((len(rows), w.d))
    for c0 in range(0, w.inter, chunk):
        c1 = min(w.inter, c0 + chunk)
        out += O.dense_ffn(xr, to64(wg[c0:c1]), to64(wu[c0:c1]), to64(wd[:, c0:c1]), w.beta, w.beta_u)
    return out


def _check(got, ref):
    m = float(np.abs(got - ref).max())
    r = rel_l2(got, ref)
    assert m <= BF16_MAX_ABS and r <= BF16_REL_L2, (m, r)


@pytest.mark.parametrize("bt", [333, 1, 17, 200])
def test_dense_ffn_small_matches_oracle(bt):
    w = FFN_WORKLOADS["dense_ffn_small"]
    x, wg, wu, wd = make_ffn_inputs(w, "cuda", bt)
    ffn = DenseFFN(w.d, w.inter, wg, wu, wd, max_bt=333, beta=w.beta, beta_u=w.beta_u)
    out = ffn.forward(x)
    torch.cuda.synchronize()
    assert ffn.sync_status() == 0
    _check(to64(out), _oracle_rows(x, wg, wu, wd, w, np.arange(bt)))
    again = ffn.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(again, out)
    ffn.close()


def test_dense_ffn_full_width_sampled_rows():
    """d = 7168, intermediate 33 792 (727 M parameters), 300 tokens; sampled rows."""
    w = FFN_WORKLOADS["dense_ffn_bt8192"]
    x, wg, wu, wd = make_ffn_inputs(w, "cuda", 300)
    ffn = DenseFFN(w.d, w.inter, wg, wu, wd, max_bt=300, beta=w.beta, beta_u=w.beta_u)
    out = ffn.forward(x)
    torch.cuda.synchronize()
    assert ffn.sync_status() == 0
    rows = np.array([0, 1, 150, 191, 192, 299])
    _check(to64(out[rows]), _oracle_rows(x, wg, wu, wd, w, rows))
    ffn.close()


def test_dense_ffn_argument_errors():
    w = FFN_WORKLOADS["dense_ffn_small"]
    x, wg, wu, wd = make_ffn_inputs(w, "cuda", 16)
    ffn = DenseFFN(w.d, w.inter, wg, wu, wd, max_bt=16)
    out = torch.empty((16, w.d), dtype=torch.bfloat16, device="cuda")
    assert L.lmoe_ffn_forward(ffn.ffn, x.data_ptr(), 17, out.data_ptr()) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_ffn_forward(ffn.ffn, x.data_ptr(), 8, x.data_ptr()) == L.LMOE_ERR_INVALID_ARG
    assert L.lmoe_ffn_forward(ffn.ffn, x.data_ptr(), 0, 0) == L.LMOE_OK
    with pytest.raises(LmoeError) as ei:
        DenseFFN(w.d, w.inter + 32, wg, wu, wd, max_bt=16)
    assert ei.value.status == L.LMOE_ERR_UNSUPPORTED
    with pytest.raises(LmoeError) as ei:
        DenseFFN(w.d, w.inter, wg.cpu(), wu, wd, max_bt=16)
    assert ei.value.status == L.LMOE_ERR_INVALID_ARG
    ffn.close()
