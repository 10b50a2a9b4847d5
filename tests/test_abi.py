"""The C ABI library loads, exports what the header declares, and checks arguments (no GPU)."""
import ast
import os
import re

import numpy as np
import pytest

import synth
import latent_sparse_moe_router_b300 as ext
from oracle import record

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "edge0_moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(edge0_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = ext.lib()
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ext.EXPORTED)


def test_record_sizes():
    assert ext.edge0_expert_record_bytes(1792, 640) == 1_935_360 + 12
    assert ext.edge0_expert_record_stride(1792, 640) == 1_935_616
    assert ext.edge0_expert_record_bytes(1280, 640) == 1_382_412
    assert ext.edge0_expert_record_bytes(1792, 640) == record.record_bytes(1792, 640)
    assert ext.edge0_expert_record_bytes(100, 640) == 0         # latent not a multiple of 256
    assert ext.edge0_expert_record_bytes(1792, 70) == 0


def test_host_packer_matches_record_layout():
    for L, F, e in ((256, 128, 3), (1280, 640, 511)):
        codes, scales, glob = synth.expert_bytes(9, 1, e, L, F)
        glob = np.float32([0.75, 1.5, -2.0])
        rec = ext.edge0_pack_expert_host(codes, scales, glob, L, F)
        c, s, g = record.read_record(rec, L, F)
        assert np.array_equal(c, codes) and np.array_equal(s, scales) and np.array_equal(g, glob)


def test_argument_checks_without_gpu():
    lib = ext.lib()
    assert lib.edge0_pack_expert_host(None, None, None, 256, 128, None) == ext.EDGE0_ERR_INVALID_ARG
    assert lib.edge0_moe_create(None, None) == ext.EDGE0_ERR_INVALID_ARG
    assert lib.edge0_moe_forward(None, None, None, 1, None) == ext.EDGE0_ERR_INVALID_ARG
    assert lib.edge0_moe_get_error(None) == ext.EDGE0_ERR_INVALID_ARG
    assert lib.edge0_residual_rmsnorm(None, None, None, -1, 2560, 1e-6, None) == ext.EDGE0_ERR_INVALID_ARG
    assert ext.edge0_status_string(ext.EDGE0_ERR_TIMEOUT) == "device wait timed out"
    lib.edge0_moe_destroy(None)


def test_create_rejects_bad_shapes_before_touching_the_device():
    d = ext.edge0_moe_desc(2560, 1000, 512, 10, 640, 16, 16, 16, 16, None, 256, 1935616, 256)
    import ctypes
    h = ctypes.c_void_p()
    assert ext.lib().edge0_moe_create(ctypes.byref(d), ctypes.byref(h)) == ext.EDGE0_ERR_INVALID_ARG
    d.latent, d.top_k = 1792, 17
    assert ext.lib().edge0_moe_create(ctypes.byref(d), ctypes.byref(h)) == ext.EDGE0_ERR_INVALID_ARG
    assert h.value is None


def test_create_rejects_bad_groups_before_touching_the_device():
    import ctypes
    stride = ext.edge0_expert_record_stride(1792, 640)
    h = ctypes.c_void_p()
    for n_groups, labels, shared in ((17, 256, 0), (-1, 256, 0), (2, None, 0), (2, 258, 0), (2, 256, 2),
                                     (8, 256, -1), (16, 256, 0)):   # 16 x 1792 > 16384 latent columns
        d = ext.edge0_moe_desc(2560, 1792, 512, 10, 640, 16, 256, 256, 256, None, 256, stride, 256,
                               n_groups, labels, shared)
        assert ext.lib().edge0_moe_create(ctypes.byref(d), ctypes.byref(h)) == ext.EDGE0_ERR_INVALID_ARG
        assert h.value is None


def _imports(path):
    tree = ast.parse(open(path).read())
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.add(node.module.split(".")[0])
    return out


def test_oracle_and_product_share_no_code():
    pkg = os.path.join(ROOT, "latent_sparse_moe_router_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                assert "oracle" not in _imports(os.path.join(dirpath, f)), f
            if f.endswith((".cu", ".cuh", ".h")):
                assert "oracle" not in open(os.path.join(dirpath, f)).read().lower(), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith(".py"):
            imps = _imports(os.path.join(ROOT, "oracle", f))
            assert "latent_sparse_moe_router_b300" not in imps and "synth" not in imps, f
