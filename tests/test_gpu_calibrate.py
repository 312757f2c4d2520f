"""GPU parity of the R_K and R_V calibrations (oscar_calibrate_rk, _rv) against the oracle.

The calibration is unique once the eigenvalues are distinct (descending order,
sign convention), so R_K is compared entry by entry: the GPU computes Sigma and
the eigenvectors in float64 (one-sided Jacobi) and writes float32; the oracle
uses float64 and numpy's eigensolver.  Tolerance 1e-5 on entries of magnitude
about 1/sqrt(D): the Jacobi stops after the sweep in which the largest |cosine|
between two rotated columns of Sigma V is at most 1e-15 (or after 40 sweeps,
which sets OSCAR_DEV_NOT_CONVERGED); a residual cosine c between columns i and j
turns the eigenvector pair by about c / delta_ij, delta_ij their relative
eigenvalue gap, so with the smallest relative gaps of these inputs
(3e-7 .. 5e-6) the eigenvector error is below 1e-8, far inside the tolerance,
to which float32 rounding of R (6e-8 relative) adds little.  The diagonal case
is exact up to rounding.  R_V uses the same fit on the value covariance weighted
by score energy; its inputs here have gaps in the same range.  A non-finite
calibration row is flagged (OSCAR_DEV_NONFINITE) instead of passing silently."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


def _gpu_calibrate(q: np.ndarray):
    d = q.shape[1]
    qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    out = torch.full((d, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.calibrate_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.calibrate_rk(qt, out, ws, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(st.item())


@pytest.mark.parametrize("d", [128, 256])
def test_calibrate_diagonal_case(d):
    rng = np.random.default_rng(51)
    scale = rng.permutation(np.arange(1, d + 1)).astype(np.float32)
    q = np.zeros((2 * d, d), dtype=np.float32)
    for i in range(d):
        q[2 * i, i] = scale[i]
        q[2 * i + 1, i] = -scale[i]
    got, st = _gpu_calibrate(q)
    assert st == 0
    assert np.abs(got - O.calibrate_rk(q)).max() <= 1e-6


@pytest.mark.parametrize("d,n", [(128, 4096), (256, 3000), (512, 2048)])
def test_calibrate_matches_oracle(d, n):
    rng = np.random.default_rng(d + n)
    ch = rng.choice(d, max(1, round(0.02 * d)), replace=False)
    q = S.activations(rng, (n, d), ch, kind="t3")
    got, st = _gpu_calibrate(q)
    assert st == 0
    ref = O.calibrate_rk(q)
    assert np.abs(got - ref).max() <= 1e-5, np.abs(got - ref).max()
    assert np.abs(got @ got.T - np.eye(d)).max() <= 1e-5


def _gpu_calibrate_rv(q, k, v):
    d = q.shape[1]
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda() for x in (q, k, v))
    out = torch.full((d, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.calibrate_rv_workspace_bytes(d, k.shape[0]), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.calibrate_rv(qt, kt, vt, out, ws, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(st.item())


@pytest.mark.parametrize("d", [128, 256])
def test_calibrate_rv_diagonal_case(d):
    # channel i: values +-a_i e_i with key e_i, queries sig_j e_j: Sigma_V is
    # diagonal and the weights, not the value magnitudes, set the order
    rng = np.random.default_rng(70 + d)
    perm = rng.permutation(d)
    a = (1.0 + np.arange(d) / d).astype(np.float32)
    sig = ((perm + 1.0) / a).astype(np.float32)
    q = np.diag(sig)
    k = np.repeat(np.eye(d, dtype=np.float32), 2, axis=0)
    v = np.repeat(np.diag(a), 2, axis=0) * np.tile(np.float32([1.0, -1.0]), d)[:, None]
    got, st = _gpu_calibrate_rv(q, k, v)
    assert st == 0
    assert np.abs(got - O.calibrate_rv(q, k, v)).max() <= 1e-6


@pytest.mark.parametrize("d,nq,nkv", [(128, 4096, 3000), (256, 3000, 2500), (512, 2048, 2100)])
def test_calibrate_rv_matches_oracle(d, nq, nkv):
    rng = np.random.default_rng(d + nq + nkv)
    ch = rng.choice(d, max(1, round(0.02 * d)), replace=False)
    q = S.activations(rng, (nq, d), ch, kind="t3")
    k = S.activations(rng, (nkv, d), ch, kind="t3")
    v = S.activations(rng, (nkv, d), ch, kind="t3")
    got, st = _gpu_calibrate_rv(q, k, v)
    assert st == 0
    ref = O.calibrate_rv(q, k, v)
    assert np.abs(got - ref).max() <= 1e-5, np.abs(got - ref).max()
    assert np.abs(got @ got.T - np.eye(d)).max() <= 1e-5


@pytest.mark.parametrize("d", [128, 512])
def test_calibrate_nonfinite_row_is_flagged(d):
    rng = np.random.default_rng(d + 5)
    q = rng.standard_normal((2000, d)).astype(np.float32)
    q[17, 3] = np.nan
    qt = torch.from_numpy(q).cuda()
    out = torch.empty((d, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.calibrate_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.calibrate_rk(qt, out, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & K.DEV_NONFINITE
    # the same rows without the NaN calibrate cleanly
    q[17, 3] = 0.5
    st.zero_()
    K.calibrate_rk(torch.from_numpy(q).cuda(), out, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    R = out.cpu().numpy().astype(np.float64)
    assert np.abs(R @ R.T - np.eye(d)).max() < 1e-5
