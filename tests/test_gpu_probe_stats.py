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
    # relative) the other way, which moves its row's outputs by |L| 2^-8 |z|.
    # So: the 2-ulp rule everywhere but a 1e-4 fraction of the elements, and
    # every element within that rule plus the one-ulp propagation bound.
    g = out.double().cpu().numpy()
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    strict = 2.0 * F.bf16_ulp(np.maximum(np.abs(ref), 2.0 ** -6 * rms))
    err = np.abs(g - ref)
    assert (err > strict).mean() <= 1e-4, f"sampler K{K}: {(err > strict).sum()} elements beyond 2 bf16 ulps"
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
