"""Host-side tests of the C ABI: the library loads without a GPU, exports every
function include/nc.h declares, and rejects bad arguments before touching the
device."""
import ctypes

import pytest

import dense_gpt_transformer_fwd_b300 as ncp
from dense_gpt_transformer_fwd_b300 import build as nc_build
import nc_inputs


@pytest.fixture(scope="module")
def L():
    nc_build.build()
    return ncp.lib()


def test_header_functions_all_exported(L):
    names = ncp.header_functions()
    assert "nc_model_create" in names and "nc_prefill" in names and "nc_decode_step" in names
    assert "nc_kv_reset" in names
    for n in names:
        assert hasattr(L, n), f"libnc.so does not export {n}"


def test_status_strings(L):
    for code in range(9):
        s = L.nc_status_string(code)
        assert isinstance(s, bytes) and s
    assert L.nc_status_string(0) == b"ok"


def _cfg(**kw):
    sh = nc_inputs.SHAPES["tiny"]
    c = ncp.make_config(sh, 1, 80)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _create(L, cfg, weights_ptr=ctypes.c_void_p(1)):
    h = ctypes.c_void_p(123)
    st = L.nc_model_create(ctypes.byref(cfg), weights_ptr, ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("field,value,want", [
    ("n_layer", 0, 1), ("d_model", 0, 1), ("n_head", 0, 1), ("vocab", 0, 1),
    ("max_batch", 0, 1), ("max_seq", 0, 1), ("dtype", 7, 1), ("softcap", 0.0, 1),
    ("rope_base", -1.0, 1), ("n_kv_head", 3, 1), ("n_kv_head", 0, 1), ("window", -1, 1),
    ("head_dim", 96, 2),
])
def test_create_rejects_bad_config_without_gpu(L, field, value, want):
    st, h = _create(L, _cfg(**{field: value}))
    assert st == want
    assert h.value is None          # *out cleared on failure


def test_create_bf16_shape_rules(L):
    c = ncp.make_config(nc_inputs.SHAPES["d12"], 1, 16)
    c.head_dim = 64
    assert _create(L, c)[0] == 2
    c = ncp.make_config(nc_inputs.SHAPES["d12"], 1, 16)
    c.n_head = 5                    # (n_head + 2) * 128 not a multiple of 256
    assert _create(L, c)[0] == 2


def test_create_null_arguments(L):
    assert L.nc_model_create(None, ctypes.c_void_p(1), ctypes.byref(ctypes.c_void_p())) == 1
    assert _create(L, _cfg(), ctypes.c_void_p())[0] == 1
    assert L.nc_model_create(ctypes.byref(_cfg()), ctypes.c_void_p(1), None) == 1


def test_calls_on_null_model(L):
    P = ctypes.c_void_p
    assert L.nc_prefill(None, P(1), 1, 1, P(1), 0, None) == 1
    assert L.nc_decode_step(None, P(1), 1, P(1), None) == 1
    assert L.nc_kv_reset(None, None) == 1
    assert L.nc_sync_status(None, None) == 1
    assert L.nc_launch_count(None) == -1
    assert L.nc_set_wait_limit(None, 10**9) == 1
    L.nc_model_destroy(None)
