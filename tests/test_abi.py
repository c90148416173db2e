"""The C-ABI library loads without a GPU, exports every function include/rq.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes as C
import os
import re

import pytest

import __graft_entry__
from rq_transformer_frame_gb300 import binding, configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "rq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rq_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.rq_abi_version() == 1
    assert lib.rq_status_string(0) == b"ok"
    assert b"token" in lib.rq_status_string(2)


def test_weight_struct_matches_header():
    src = open(os.path.join(ROOT, "include", "rq.h")).read()
    body = src[src.index("typedef struct {\n  const void *emb"):]
    body = body[:body.index("} rq_weights;")]
    names = re.findall(r"\*\s*([a-z_0-9]+)", body)
    assert names == binding.WEIGHT_FIELDS


def test_config_struct_matches_header():
    src = open(os.path.join(ROOT, "include", "rq.h")).read()
    body = src[src.index("typedef struct {\n  int32_t batch;"):]
    body = body[:body.index("} rq_config;")]
    names = re.findall(r"(?:int32_t|float)\s+([a-z_]+);", body)
    assert names == [n for n, _ in binding.RqConfig._fields_]


def _null_weights():
    return binding.RqWeights(**{n: None for n in binding.WEIGHT_FIELDS})


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 48, binding.RQ_ERR_ARG),      # dim != heads * head_dim
    ("batch", 0, binding.RQ_ERR_ARG),
    ("weight_dtype", 7, binding.RQ_ERR_ARG),
])
def test_create_rejects_bad_config_on_host(lib, field, value, status):
    c = binding.make_config(configs.TINY)
    setattr(c, field, value)
    h = C.c_void_p()
    st = lib.rq_create(C.byref(c), C.byref(_null_weights()), None, C.byref(h))
    assert st == status
    assert not h.value
    assert len(lib.rq_last_error(None)) > 0


def test_create_rejects_unaligned_weights_on_host(lib):
    c = binding.make_config(configs.TINY)
    w = binding.RqWeights(**{n: 4096 * (i + 1) + 4 for i, n in enumerate(binding.WEIGHT_FIELDS)})
    h = C.c_void_p()
    assert lib.rq_create(C.byref(c), C.byref(w), None, C.byref(h)) == binding.RQ_ERR_ARG
    assert not h.value


def test_calls_on_null_handle_are_errors(lib):
    assert lib.rq_reset(None, -1) == binding.RQ_ERR_ARG
    assert lib.rq_step(None, None, None, None) == binding.RQ_ERR_ARG
    assert lib.rq_frame_kernel_count(None) == 0
    lib.rq_destroy(None)


def test_band_row_bytes_and_quantizer_arguments_on_host(lib):
    # codes, then one f32 scale per 32 values
    assert lib.rq_band_row_bytes(binding.RQ_Q8, 4096) == 4096 + 512
    assert lib.rq_band_row_bytes(binding.RQ_Q4, 4096) == 2048 + 512
    assert lib.rq_band_row_bytes(binding.RQ_BF16, 64) == 128
    assert lib.rq_band_row_bytes(binding.RQ_Q4, 48) == 0  # not a multiple of 32
    bad = [(binding.RQ_Q4, binding.RQ_BF16, 2, 48), (binding.RQ_BF16, binding.RQ_BF16, 2, 64),
           (binding.RQ_Q8, 9, 2, 64), (binding.RQ_Q8, binding.RQ_F32, -1, 64)]
    for dt, sdt, rows, cols in bad:
        assert lib.rq_quantize(dt, 16, sdt, rows, cols, 32, None) == binding.RQ_ERR_ARG
    assert set(binding.MATRIX_FIELDS) <= set(binding.WEIGHT_FIELDS)


def test_create_rejects_bands_with_short_rows_on_host(lib):
    c = binding.make_config(configs.TINY.with_(weight_dtype="q4"))  # hidden 704, not /128
    h = C.c_void_p()
    assert lib.rq_create(C.byref(c), C.byref(_null_weights()), None, C.byref(h)) == \
        binding.RQ_ERR_UNSUPPORTED
    assert not h.value


def test_new_entry_points_on_null_handle_are_errors(lib):
    assert lib.rq_set_sampling(None, 1, 0.8, 0.7, 25, 25, None) == binding.RQ_ERR_ARG
    assert lib.rq_get_rng(None, None) == binding.RQ_ERR_ARG
    assert lib.rq_prime(None, 0, 1, None, None) == binding.RQ_ERR_ARG
    assert lib.rq_replay(None, 0, 1, None) == binding.RQ_ERR_ARG
    assert lib.rq_snapshot_size(None, 0) == 0
    assert lib.rq_snapshot(None, 0, None, 0) == binding.RQ_ERR_ARG
    assert lib.rq_restore(None, 0, None, 0) == binding.RQ_ERR_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """There is no CPU fallback: without the built CUDA library the binding raises."""
    monkeypatch.setattr(binding, "LIBPATH", str(tmp_path / "librq.so"))
    monkeypatch.setattr(binding, "_LIB", None)
    with pytest.raises(RuntimeError, match="not built"):
        binding.load()
