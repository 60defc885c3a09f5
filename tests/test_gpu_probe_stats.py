"""GPU parity of LoKA Probe's online input statistics and sampler (section
III-A 1): the running mean and scatter matrix after several batches against
the oracle's Chan update in float64, and the sampled inputs Z L^T + mu
against the oracle's, drawn from the same counter-based stream."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import probe_stats as PS

import fp8_precision_recommendation_gb300 as loka

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _batches(K, sizes, seed):
    rng = np.random.default_rng(seed)
    means = rng.uniform(-1.0, 1.0, K)
    scales = rng.uniform(0.5, 2.0, K)
    out = []
    for i, b in enumerate(sizes):
        x = W.random_bf16((b, K), seed=seed * 100 + i, outlier_frac=0.01).float().numpy()
        out.append(torch.from_numpy(x * scales + means).to(torch.bfloat16))
    return out


def _check_stats(st, n, mu, S, what):
    assert st.n == n
    mg, sg = st.mu.cpu().numpy(), st.scatter.cpu().numpy()
    d = np.sqrt(np.outer(np.diag(S), np.diag(S)))
    assert np.abs(mg - mu).max() <= 1e-5 * np.sqrt(np.diag(S).max() / n) + 1e-9, f"{what}: mean"
    err = np.abs(sg - S)
    assert (err <= 1e-4 * d + 1e-6).all(), f"{what}: scatter, worst {(err / (d + 1e-30)).max():.2e} of scale"
    # the batch scatter accumulates in fp32 on the tensor cores over up to
    # 4096 products per split-K group (the pages accumulate in "higher
    # precision, e.g. FP32"): worst case 4096 * 2^-23 = 4.9e-4 relative, a
    # few 1e-5 measured on 65536 x 512 with 1% outliers
    assert np.linalg.norm(sg - S) <= 1e-4 * np.linalg.norm(S), f"{what}: normwise"


@pytest.mark.parametrize("K", [128, 512, 2048])
def test_statistics_over_ragged_batches(lib, K):
    # batch sizes: ragged (zero-padded split-K groups), one row, several full groups
    sizes = [300, 1, 4096, 20000] if K < 2048 else [300, 5000]
    st = loka.InputStats(K, DEV)
    n, mu, S = 0, np.zeros(K), np.zeros((K, K))
    for i, xb in enumerate(_batches(K, sizes, seed=K)):
        st.update(xb.to(DEV))
        n, mu, S = PS.stats_update(n, mu, S, xb.float().numpy())
        torch.cuda.synchronize()
        assert loka._loka.loka_device_status() == 0
        _check_stats(st, n, mu, S, f"K{K} after batch {i}")
    cov, ref = st.covariance().cpu().numpy(), PS.covariance(n, S)
    scale = np.sqrt(np.outer(np.diag(ref), np.diag(ref)))
    assert (np.abs(cov - ref) <= 1e-4 * scale).all()


def test_statistics_full_size_batch(lib):
    inp = W.rec_mlp()
    st = loka.InputStats(inp.K, DEV)
    st.update(inp.x.to(DEV))
    torch.cuda.synchronize()
    n, mu, S = PS.stats_update(0, np.zeros(inp.K), np.zeros((inp.K, inp.K)), inp.x.float().numpy())
    _check_stats(st, n, mu, S, "65536 x 512")


@pytest.mark.parametrize("K,B", [(128, 1000), (512, 4096)])
def test_sampler_against_oracle_stream(lib, K, B):
    rng = np.random.default_rng(K)
    A = rng.standard_normal((K, K)) / np.sqrt(K)
    sigma = A @ A.T + 0.2 * np.eye(K)
    L = torch.from_numpy(np.linalg.cholesky(sigma)).to(torch.bfloat16)
    mu = torch.from_numpy(rng.uniform(-1, 1, K)).to(torch.bfloat16)
    out = loka.sample_inputs(mu.to(DEV), L.to(DEV), B, seed=11)
    torch.cuda.synchronize()
    # the oracle's stream, rounded to bf16 as the device rounds its normals
    Z, _ = PS.sample_inputs(np.zeros(K), np.eye(K), B, seed=11)
    Zb = torch.from_numpy(Z).to(torch.bfloat16).double().numpy()
    ref = Zb @ L.double().numpy().T + mu.double().numpy()[None, :]
    # The device evaluates Box-Muller in fp32, the oracle in fp64: a normal
    # within rounding distance of a bf16 midpoint may round one ulp (2^-8
    # relative) the other way, which moves its row's outputs by at most
    # 2^-8 sum_k |z_k| |L_jk|.  Every element: the 2-ulp rule plus that
    # propagation bound.
    g = out.double().cpu().numpy()
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    strict = 2.0 * F.bf16_ulp(np.maximum(np.abs(ref), 2.0 ** -6 * rms))
    err = np.abs(g - ref)
    prop = 2.0 ** -8 * (np.abs(Zb) @ np.abs(L.double().numpy()).T)
    assert (err <= strict + prop).all(), f"sampler K{K}: beyond the one-ulp propagation bound"
    # the samples carry the requested second moments
    if B >= 4096:
        c = np.cov(out.double().cpu().numpy(), rowvar=False)
        LL = L.double().numpy() @ L.double().numpy().T
        assert np.abs(c - LL).max() <= 0.15 * np.abs(LL).max()


@pytest.mark.parametrize("K", [128, 512])
def test_cholesky_factor_against_oracle(lib, K):
    st = loka.InputStats(K, DEV)
    n, mu, S = 0, np.zeros(K), np.zeros((K, K))
    for xb in _batches(K, [3000, 5000], seed=40 + K):
        st.update(xb.to(DEV))
        n, mu, S = PS.stats_update(n, mu, S, xb.float().numpy())
    L, m = st.factor(eps_rel=1e-6)
    torch.cuda.synchronize()
    Lo = PS.cholesky_factor(n, S, 1e-6)
    Lg = L.double().cpu().numpy()
    assert np.array_equal(np.triu(Lg, 1), np.zeros_like(Lg))
    # backward error, per element: bf16 storage (8 significant bits) moves
    # each L_ik by at most 2^-8 |L_ik|, so a product term by 2^-7 |L_ik L_jk|
    # (plus 2^-16 second order), and the fp32 factorization adds
    # K 2^-24 |L||L^T|
    A = PS.covariance(n, S)
    A = A + 1e-6 * np.trace(A) / K * np.eye(K)
    absLL = np.abs(Lg) @ np.abs(Lg).T
    assert (np.abs(Lg @ Lg.T - A) <= (2.0 ** -7 + 2.0 ** -16 + K * 2.0 ** -24) * absLL).all(), f"K{K}: residual"
    # bf16 storage (2 ulps) and the fp32 factorization's rounding
    tol = 2.0 * F.bf16_ulp(np.abs(Lo)) + 1e-3 * np.abs(Lo).max()
    assert (np.abs(Lg - Lo) <= tol).all(), f"K{K}: worst {np.abs(Lg - Lo).max():.3e}"
    assert (np.abs(m.double().cpu().numpy() - mu) <= 2.0 * F.bf16_ulp(np.abs(mu)) + 1e-6).all()


def test_cholesky_rejects_an_indefinite_covariance(lib):
    st = loka.InputStats(128, DEV)
    st.c.n = 10
    st.scatter.copy_(torch.diag(torch.tensor([1.0, -1.0] + [1.0] * 126, dtype=torch.float64)))
    with pytest.raises(loka._loka.LokaError) as e:
        st.factor(eps_rel=0.0)
    assert e.value.status == loka._loka.LOKA_ERR_NUMERIC


def test_probe_on_learned_inputs(lib):
    # the probe loop on the device: learn a layer's input statistics, factor
    # the covariance, sample inputs from it and measure the FP8 error on them
    K = 512
    st = loka.InputStats(K, DEV)
    for xb in _batches(K, [8192, 8192], seed=5):
        st.update(xb.to(DEV))
    L, m = st.factor(eps_rel=1e-6)
    xs = loka.sample_inputs(m, L, 4096, seed=2)
    w = W.random_bf16((256, K), seed=3, var=1.0 / K).to(DEV)
    err = loka.quant_error(xs, w, None, W.SCALE_ROW)
    assert 1e-3 < err["rel_err_fro"] < 0.1 and np.isfinite(err["mere"])


# ------------------------------------------------------- the weight model
from oracle import probe_weights as PW


def _weights(R, C, count, seed):
    # a slowly drifting weight with row- and column-correlated noise
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((R, C)) / np.sqrt(C)
    rmix = np.eye(R) + 0.3 * rng.standard_normal((R, R)) / np.sqrt(R)
    cmix = np.eye(C) + 0.3 * rng.standard_normal((C, C)) / np.sqrt(C)
    out = []
    for t in range(count):
        w = base * (1 + 0.01 * t) + 0.05 * rmix @ rng.standard_normal((R, C)) @ cmix.T / np.sqrt(C)
        out.append(torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16))
    return out


@pytest.mark.parametrize("R,C", [(64, 96), (256, 512), (1024, 2048)])
def test_weight_model_update_against_oracle(lib, R, C):
    wm = loka.WeightModel(R, C, DEV)
    st = None
    for t, w in enumerate(_weights(R, C, 6, seed=R + C)):
        wm.update(w.to(DEV), momentum=0.9, eps_rel=1e-6)
        st = PW.weight_update(st, w.float().numpy(), 0.9, 1e-6)
        torch.cuda.synchronize()
        assert loka._loka.loka_device_status() == 0
        assert wm.n == st.n == t + 1
        M, U, V = (a.double().cpu().numpy() for a in (wm.mean, wm.U, wm.V))
        # fp32 moving average of the mean; fp32 factorizations, solves and
        # products for the covariances (the oracle is fp64)
        assert np.abs(M - st.M).max() <= 1e-5 * np.abs(st.M).max(), f"update {t}: mean"
        for name, a, b in (("U", U, st.U), ("V", V, st.V)):
            assert np.linalg.norm(a - b) <= 1e-4 * np.linalg.norm(b), f"update {t}: {name} normwise"
            assert np.abs(a - b).max() <= 2e-4 * np.abs(b).max(), f"update {t}: {name}"
        assert abs(np.trace(U) - R) <= 1e-4 * R


def test_weight_sampler_against_oracle(lib):
    R, C = 128, 256
    wm = loka.WeightModel(R, C, DEV)
    for w in _weights(R, C, 5, seed=9):
        wm.update(w.to(DEV), momentum=0.9, eps_rel=1e-6)
    out = wm.sample(seed=21, eps_rel=1e-6)
    torch.cuda.synchronize()
    st = PW.WeightStats(wm.n, *(a.double().cpu().numpy() for a in (wm.mean, wm.U, wm.V)))
    Z, ref = PW.weight_sample(st, 1e-6, 21)
    g = out.double().cpu().numpy()
    # per element: the 2-ulp rule of the bf16 output, plus the fp32 path's
    # rounding (Box-Muller, the two factorizations and the two products, a
    # few hundred ulps of fp32 on the terms |L_U| |Z| |L_V|^T)
    LU = PW.reg_cholesky(st.U, 1e-6)
    LV = PW.reg_cholesky(st.V, 1e-6)
    terms = np.abs(LU) @ np.abs(Z) @ np.abs(LV).T
    rms = np.sqrt(np.mean(ref * ref))
    tol = 2.0 * F.bf16_ulp(np.maximum(np.abs(ref), 2.0 ** -6 * rms)) + 1e-5 * terms
    err = np.abs(g - ref)
    assert (err <= tol).all(), f"{int((err > tol).sum())} elements beyond the bound; worst {err.max():.3e}"


def test_weight_model_rejects_an_indefinite_factor(lib):
    wm = loka.WeightModel(32, 32, DEV)
    wm.update(W.random_bf16((32, 32), seed=1).to(DEV))
    wm.U.copy_(-torch.eye(32, device=DEV))
    with pytest.raises(loka._loka.LokaError) as e:
        wm.sample(seed=1, eps_rel=0.0)
    assert e.value.status == loka._loka.LOKA_ERR_NUMERIC


def test_probe_on_learned_inputs_and_weights(lib):
    # the whole probe loop on the device (LoKA section III-A): learn a
    # layer's input statistics and its weight model, sample both, and
    # measure the FP8 error of the layer on the samples
    K, N = 512, 256
    st = loka.InputStats(K, DEV)
    for xb in _batches(K, [8192, 8192], seed=7):
        st.update(xb.to(DEV))
    L, m = st.factor(eps_rel=1e-6)
    wm = loka.WeightModel(N, K, DEV)
    for w in _weights(N, K, 8, seed=8):
        wm.update(w.to(DEV), momentum=0.9)
    xs = loka.sample_inputs(m, L, 4096, seed=2)
    ws = wm.sample(seed=3)
    err = loka.quant_error(xs, ws, None, W.SCALE_ROW)
    assert 1e-3 < err["rel_err_fro"] < 0.1 and np.isfinite(err["mere"])
