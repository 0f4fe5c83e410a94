"""The C-ABI library builds, loads and exports every symbol include/hq.h
declares; host-only entry points agree with the oracle (no GPU needed)."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "hq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(hq_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def hqlib():
    from weights_hq_encode_gb300 import build
    build.build()
    from weights_hq_encode_gb300 import hq
    return hq


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("hq_encode", "hq_decode", "hq_decode_qk", "hq_make_signs", "hq_status_string",
              "hq_num_groups", "hq_encode_workspace_bytes", "hq_decode_qk_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(hqlib):
    import ctypes
    L = ctypes.CDLL(hqlib.library_path())
    for n in _declared_functions():
        assert hasattr(L, n), n
    assert set(hqlib.EXPORTED) >= set(_declared_functions())


def test_host_entry_points(hqlib, oracle):
    for seed, seg in ((0, 0), (20, 0), (21, 31), (2**64 - 1, 2**40 + 3)):
        assert hqlib.hq_make_signs(seed, seg) == [int(v) for v in oracle.make_signs(seed, seg)]
    for sd, ss, layer in ((20, 21, 0), (20, 21, 31), (1, 2**63 + 5, 7)):
        want = oracle.make_signs(sd, 0) ^ oracle.make_signs(ss, layer)
        assert hqlib.hq_make_layer_signs(sd, ss, layer) == [int(v) for v in want]
    assert hqlib.hq_num_groups(0) == 0
    assert hqlib.hq_num_groups(1) == 1 and hqlib.hq_num_groups(32) == 1
    assert hqlib.hq_num_groups(33) == 2
    assert hqlib.hq_num_groups(4194304) == oracle.n_groups(4194304)
    assert hqlib.hq_encode_workspace_bytes(129) >= 8 + 8 * 2
    assert hqlib.hq_decode_qk_workspace_bytes(16, 32) == 16 * 32 * 128 * 4
    assert hqlib.hq_status_string(8) == "corrupt stream"
    assert hqlib.hq_status_string(0) == "ok"


def test_noalloc_limit_fits_the_built_in_scratch(hqlib):
    # the encoder workspace of the largest call hq_encode_noalloc accepts must
    # fit the ~1 MiB array compiled into the library (8 bytes of header plus 8
    # per 32-tile block, rounded up to 256 bytes)
    need = hqlib.hq_encode_workspace_bytes(hqlib.HQ_NOALLOC_MAX_TILES)
    assert need <= ((8 + 8 * (hqlib.HQ_NOALLOC_MAX_TILES // 32)) + 255) // 256 * 256
    assert need <= (1 << 20) + 256


def test_params_layout(hqlib):
    import ctypes
    # the ctypes mirror must match the C struct: 4+4+4+4+8+8+8+8+4+4+8 = 64 bytes
    assert ctypes.sizeof(hqlib.hq_params) == 64
    assert hqlib.hq_params.d_rot.offset == 56
    assert hqlib.hq_params.d_signs.offset == 32


def test_calibration_layout(hqlib):
    import ctypes
    # float, int32, double, int32, int32 -> 4+4+8+4+4 = 24 bytes, bps at offset 8
    assert ctypes.sizeof(hqlib.hq_calibration) == 24
    assert hqlib.hq_calibration.bps.offset == 8
    assert hqlib.hq_calibration.evaluations.offset == 20
