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
