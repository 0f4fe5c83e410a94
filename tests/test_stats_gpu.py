"""Per-vector unbiasedness of the fused GPU scores (HyperQuant summary,
Method 4 and the closing section): hq_decode_qk over 64 dither seeds, sign
diagonal fixed, against q.K of the exact bf16 input."""
import numpy as np
import pytest
import torch

from _cases import calibration

pytestmark = pytest.mark.gpu
P_T63_GT3 = 0.00387


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


def test_fused_scores_unbiased_over_64_seeds(hq):
    from weights_hq_encode_gb300 import inputs as I
    C = I.SCORES
    cal = calibration()["kv_cache_8b"]["E8"]["3.0"]
    n_kv, T, B, Hq = 2, 1024, 4, 8
    K = I.scores_keys("cuda", tokens=T)[:n_kv].contiguous()
    q = I.scores_queries("cuda", batch=B, q_heads=Hq)
    exact = torch.einsum("bgkd,ktd->bgkt", q.double().view(B, n_kv, Hq // n_kv, 128).transpose(1, 2),
                         K.double()).transpose(1, 2).reshape(B, Hq, T)
    m = [a ^ b for a, b in zip(hq.hq_make_signs(C["sign_seed"], 0),
                                hq.hq_make_signs(C["layer_sign_seed"], 0))]
    signs = torch.from_numpy(np.asarray(m, np.uint32).view(np.int32).reshape(1, 4)).cuda()
    n = n_kv * T
    ws = torch.empty(hq.hq_decode_qk_workspace_bytes(B, Hq), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    errs = []
    for seed in C["dither_seeds"]:
        p = hq.make_params(8, cal["k"], cal["alpha"], 1, seed, signs, n)
        enc = hq.encode(K, p)
        scores = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
        assert hq.hq_decode_qk(p, enc.stream, enc.total_words, enc.offsets, n_kv, T,
                               q.view(torch.int16), B, Hq, scores, ws, st) == 0
        errs.append((scores.double() - exact).cpu().numpy())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    E = np.stack(errs)
    ns = E.shape[0]
    t = E.mean(0) / (E.std(0, ddof=1) / np.sqrt(ns))
    frac = np.mean(np.abs(t) > 3)
    assert 0.25 * P_T63_GT3 <= frac <= 2.5 * P_T63_GT3, frac
    seed_means = E.reshape(ns, -1).mean(1)
    z = seed_means.mean() / (seed_means.std(ddof=1) / np.sqrt(ns))
    assert abs(z) < 4, z
