"""GPU rate calibration against the CPU oracle.

HyperQuant summary, Method 2 (alpha calibrated so that the codes fit) and
Method 3 (realized rate within about 0.01 bps of the target, k per rate).
hq_payload_bits must equal the oracle's payload size bit for bit (both count
the Rice bits of every symbol, without group padding or the index), and
hq_calibrate must retrace the oracle's bisection (oracle/calibrate.py) step
for step, so it returns the same alpha, k and realized rate."""
import numpy as np
import pytest
import torch

from _cases import Case, bits_to_torch, calibration

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq as H
    return H


def _gpu_payload(hq, c: Case):
    x = bits_to_torch(c.x_bits)
    p = c.gpu_params(hq)
    ws = torch.zeros(hq.hq_encode_workspace_bytes(c.n), dtype=torch.uint8, device="cuda")
    bits = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert hq.hq_payload_bits(p, x, c.n, bits, ws, status) == hq.HQ_OK
    torch.cuda.synchronize()
    return int(bits.item()), int(status.item())


def _tiny(oracle):
    from weights_hq_encode_gb300 import inputs as I
    x = I.bf16_bits(I.tiny_kv()).reshape(-1, 128)
    return x, oracle.make_signs(I.TINY["sign_seed"], 0).reshape(1, 4), I.TINY["dither_seed"]


@pytest.mark.parametrize("lattice,k,alpha,dither", [
    (8, 2, 1.7, 1), (8, 0, 0.4, 1), (8, 1, 0.9, 0), (8, 5, 40.0, 1),
    (4, 2, 2.5, 1), (1, 1, 3.0, 0), (8, 0, 300.0, 1),            # the last overflows some tiles
])
def test_payload_bits_equal_oracle(hq, oracle, lattice, k, alpha, dither):
    x, masks, seed = _tiny(oracle)
    x = np.concatenate([x, x[:45]])                              # ragged last group
    c = Case(x, lattice, k, alpha, dither, seed, masks, 1 << 40)
    P = c.oracle_params(oracle)
    want = oracle.payload_bits(P, c.x_bits)
    got, status = _gpu_payload(hq, c)
    assert got == want
    assert status == oracle.encode(P, c.x_bits)["status"] & ~hq.HQ_ERR_CAPACITY


def test_payload_bits_accumulate_and_empty(hq, oracle):
    x, masks, seed = _tiny(oracle)
    c = Case(x, 8, 2, 1.7, 1, seed, masks, 1 << 40)
    want = oracle.payload_bits(c.oracle_params(oracle), c.x_bits)
    xt = bits_to_torch(c.x_bits)
    p = c.gpu_params(hq)
    ws = torch.zeros(hq.hq_encode_workspace_bytes(c.n), dtype=torch.uint8, device="cuda")
    bits = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        assert hq.hq_payload_bits(p, xt, c.n, bits, ws, status) == hq.HQ_OK
    assert hq.hq_payload_bits(p, xt, 0, bits, ws, status) == hq.HQ_OK
    torch.cuda.synchronize()
    assert int(bits.item()) == 2 * want and int(status.item()) == 0
    assert hq.hq_payload_bits(p, xt, c.n, None, ws, status) == hq.HQ_ERR_INVALID


def _gpu_calibrate(hq, c: Case, target, tol, k_min, k_max):
    x = bits_to_torch(c.x_bits)
    p = c.gpu_params(hq)
    ws = torch.zeros(hq.hq_encode_workspace_bytes(c.n), dtype=torch.uint8, device="cuda")
    bits = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc, out = hq.hq_calibrate(p, x, c.n, target, tol, k_min, k_max, ws, bits, status)
    assert rc == hq.HQ_OK
    return out


def test_calibrate_tiny_equals_oracle(hq, oracle):
    from oracle import calibrate as CAL
    x, masks, seed = _tiny(oracle)
    ref = CAL.calibrate(x, oracle.E8, 3.0, 1, seed, masks, 1 << 40, ks=[2])
    c = Case(x, 8, 2, 1.0, 1, seed, masks, 1 << 40)
    out = _gpu_calibrate(hq, c, 3.0, CAL.TOL, 2, 2)
    assert out.feasible == 1
    assert (out.alpha, out.rice_k, out.bps) == (ref["alpha"], ref["k"], ref["bps"])
    # the frozen tiny entry was written by the same oracle procedure
    frozen = calibration()["tiny_kv"]["E8"]["3.0"]
    assert out.rice_k == frozen["k"]
    assert abs(out.alpha - frozen["alpha"]) <= 1e-6 * frozen["alpha"]


@pytest.mark.parametrize("lattice,target", [(8, 2.0), (4, 2.5), (1, 1.7)])
def test_calibrate_all_k_equals_oracle(hq, oracle, lattice, target):
    """k = 0..8 on two layers x 64 tokens of the KV cache (CPU-drawn)."""
    from oracle import calibrate as CAL
    from weights_hq_encode_gb300 import inputs as I
    C = I.KV8B
    xs, ms = [], []
    for layer in range(2):
        for kv in (0, 1):
            xs.append(I.bf16_bits(I.kv_slab(I.slab_seed(C["data_seed"], layer, kv),
                                            C["kv_heads"], 64)).reshape(-1, 128))
            ms.append(CAL.kv_masks(C["sign_seed"], C["layer_sign_seed"], layer))
    x, m, tps = np.concatenate(xs), np.concatenate(ms), xs[0].shape[0]
    ref = CAL.calibrate(x, lattice, target, 1, C["dither_seed"], m, tps)
    c = Case(x, lattice, 0, 1.0, 1, C["dither_seed"], m, tps)
    out = _gpu_calibrate(hq, c, target, CAL.TOL, 0, 8)
    assert out.feasible == 1
    assert (out.alpha, out.rice_k, out.bps) == (ref["alpha"], ref["k"], ref["bps"])


def test_calibrate_kv_subset_reproduces_frozen_values(hq, oracle):
    """The full calibration subset of the Llama-3.1-8B KV cache (first 256
    tokens of every layer and K/V slab, 131072 tiles) on the GPU lands on the
    (alpha, k) that the oracle froze in calibration.json.  The frozen values
    were computed on another machine, whose libm may round the draws'
    transcendental steps differently in the last place, so alpha is held to
    1e-3 here; exact agreement is the job of the on-machine tests above."""
    from oracle import calibrate as CAL
    from weights_hq_encode_gb300 import inputs as I
    C = I.KV8B
    xs, ms = [], []
    for layer in range(C["layers"]):
        for kv in (0, 1):
            xs.append(I.bf16_bits(I.kv_slab(I.slab_seed(C["data_seed"], layer, kv),
                                            C["kv_heads"], 256)).reshape(-1, 128))
            ms.append(CAL.kv_masks(C["sign_seed"], C["layer_sign_seed"], layer))
    x, m, tps = np.concatenate(xs), np.concatenate(ms), xs[0].shape[0]
    c = Case(x, 8, 0, 1.0, 1, C["dither_seed"], m, tps)
    for target in ("2.0", "3.0"):
        frozen = calibration()["kv_cache_8b"]["E8"][target]
        out = _gpu_calibrate(hq, c, float(target), CAL.TOL, 0, 8)
        assert out.feasible == 1 and out.rice_k == frozen["k"]
        assert abs(out.alpha - frozen["alpha"]) <= 1e-3 * frozen["alpha"]
        assert abs(out.bps - float(target)) <= CAL.TOL


def test_calibrate_infeasible_and_invalid(hq, oracle):
    x, masks, seed = _tiny(oracle)
    c = Case(x, 8, 2, 1.0, 1, seed, masks, 1 << 40)
    out = _gpu_calibrate(hq, c, 0.05, 0.002, 2, 2)               # below k = 2's floor
    assert out.feasible == 0
    xt = bits_to_torch(c.x_bits)
    p = c.gpu_params(hq)
    ws = torch.zeros(hq.hq_encode_workspace_bytes(c.n), dtype=torch.uint8, device="cuda")
    bits = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for args in [(3.0, 0.002, 3, 2), (3.0, 0.0, 0, 8), (-1.0, 0.002, 0, 8), (3.0, 0.002, 0, 16)]:
        rc, _ = hq.hq_calibrate(p, xt, c.n, *args, ws, bits, status)
        assert rc == hq.HQ_ERR_INVALID
