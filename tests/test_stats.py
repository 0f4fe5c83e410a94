"""Statistical pins of the oracle (no GPU).

HyperQuant summary, Method 4: subtractive dither makes the inner product
per-vector unbiased, E_U[<q, x_hat>] = <q, x> for every fixed vector x (with
the sign diagonal D fixed), which a fixed-rate quantizer lacks.  Method 3:
the realized rate lands within about 0.01 bps of the target.
"""
import numpy as np
import pytest

from _cases import calibration

# two-sided P(|t| > 3) for Student t with 63 degrees of freedom
P_T63_GT3 = 0.00387


def _scores_workload(oracle, tokens=512, batch=4, q_heads=4):
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    K = I.kv_slab(I.slab_seed(C["data_seed"], 0, 0), 1, tokens, "cpu")[0]      # [T, 128]
    q = I.scores_queries("cpu", batch=batch, q_heads=q_heads)                   # [B, Hq, 128]
    kb = I.bf16_bits(K).reshape(-1, 128)
    qb = I.bf16_bits(q)
    kf = (kb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qf = (qb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = np.einsum("bhd,td->bht", qf, kf)
    mask = (oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(C["layer_sign_seed"], 0))
    return kb, qb, exact, mask.reshape(1, 4)


def _score_errors(oracle, kb, qb, exact, mask, dither, seeds, alpha, k):
    T = kb.shape[0]
    B, Hq = qb.shape[0], qb.shape[1]
    errs = []
    for s in seeds:
        P = oracle.make_params(8, k, alpha, dither, s, mask, 1 << 40)
        enc = oracle.encode(P, kb)
        khat = oracle.decode(P, enc["stream"], enc["offsets"], T)["out"]
        sc = oracle.scores(khat, 1, T, qb, B, Hq)
        errs.append(sc.astype(np.float64) - exact)
    return np.stack(errs)                                   # [seeds, B, Hq, T]


def test_dither_makes_scores_unbiased_per_vector(oracle):
    cal = calibration()["kv_cache_8b"]["E8"]["3.0"]
    kb, qb, exact, mask = _scores_workload(oracle)
    seeds = list(range(500, 564))
    E = _score_errors(oracle, kb, qb, exact, mask, 1, seeds, cal["alpha"], cal["k"])
    n = E.shape[0]
    mean = E.mean(0)
    sd = E.std(0, ddof=1)
    t = mean / (sd / np.sqrt(n))
    frac = np.mean(np.abs(t) > 3)
    assert 0.25 * P_T63_GT3 <= frac <= 2.5 * P_T63_GT3, frac   # t_63 tail
    seed_means = E.reshape(n, -1).mean(1)                  # independent across seeds
    z = seed_means.mean() / (seed_means.std(ddof=1) / np.sqrt(n))
    assert abs(z) < 4, z
    # averaging over seeds shrinks the per-score error like 1/sqrt(n)
    rms1 = np.sqrt((E ** 2).mean())
    rms_mean = np.sqrt((mean ** 2).mean())
    assert rms_mean < 2.0 * rms1 / np.sqrt(n)


def test_without_dither_the_error_does_not_average_out(oracle):
    """Contrast: with the dither off the code is a deterministic function of x,
    so every 'seed' gives the same error and averaging removes nothing."""
    cal = calibration()["kv_cache_8b"]["E8"]["3.0"]
    kb, qb, exact, mask = _scores_workload(oracle, tokens=128)
    E = _score_errors(oracle, kb, qb, exact, mask, 0, [1, 2, 3], cal["alpha"], cal["k"])
    assert np.array_equal(E[0], E[1]) and np.array_equal(E[1], E[2])
    rms1 = np.sqrt((E[0] ** 2).mean())
    assert rms1 > 0
    assert np.sqrt((E.mean(0) ** 2).mean()) == pytest.approx(rms1)


@pytest.mark.parametrize("name,rate", [("kv_cache_8b", "2.0"), ("kv_cache_8b", "3.0")])
def test_realized_rate_on_fresh_kv_data(oracle, name, rate):
    """The frozen (alpha, k) reach the target within 0.01 bps on KV tokens that
    were not part of the calibration subset (tokens 256..383 of every slab)."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.KV8B
    c = calibration()[name]["E8"][rate]
    xs, ms = [], []
    for layer in range(C["layers"]):
        for kv in (0, 1):
            x = I.kv_slab(I.slab_seed(C["data_seed"], layer, kv), C["kv_heads"], 384, "cpu")
            xs.append(I.bf16_bits(x[:, 256:]).reshape(-1, 128))     # tokens 256..383
            ms.append(oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(C["layer_sign_seed"], layer))
    x = np.concatenate(xs)
    P = oracle.make_params(8, c["k"], c["alpha"], 1, C["dither_seed"], np.stack(ms), xs[0].shape[0])
    bps = oracle.payload_bits(P, x) / x.size
    assert abs(bps - float(rate)) < 0.01, bps


def test_calibrated_rates_recorded_within_tolerance():
    cal = calibration()
    for name, lat in cal.items():
        if name.startswith("_"):
            continue
        for lname, rates in lat.items():
            for rate, c in rates.items():
                for entry in (c if isinstance(c, list) else [c]):
                    assert abs(entry["bps"] - float(rate)) <= 0.002 + 1e-9, (name, lname, rate)


def test_compression_at_3_bps_matches_the_stated_context(oracle):
    """HyperQuant summary, Experimental results (KV cache): about 81% less memory at
    3 bps than bf16 (1 - 3/16 = 81.25%).  The whole stream (payload, group padding and
    the 64-bit group index) of fresh KV tokens at the frozen 3-bps setting
    lands within half a point of it."""
    from weights_hq_encode_gb300 import inputs as I
    C = I.KV8B
    c = calibration()["kv_cache_8b"]["E8"]["3.0"]
    xs, ms = [], []
    for layer in range(0, C["layers"], 4):
        for kv in (0, 1):
            x = I.kv_slab(I.slab_seed(C["data_seed"], layer, kv), C["kv_heads"], 384, "cpu")
            xs.append(I.bf16_bits(x[:, 256:]).reshape(-1, 128))
            ms.append(oracle.make_signs(C["sign_seed"], 0) ^ oracle.make_signs(C["layer_sign_seed"], layer))
    x = np.concatenate(xs)
    P = oracle.make_params(8, c["k"], c["alpha"], 1, C["dither_seed"], np.stack(ms), xs[0].shape[0])
    enc = oracle.encode(P, x)
    total_bits = enc["total_words"] * 32 + 64 * (oracle.n_groups(x.shape[0]) + 1)
    compression = 1 - total_bits / (x.size * 16)
    assert abs(compression - 0.8125) < 0.005, compression
