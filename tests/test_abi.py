"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before it makes
any CUDA call.  No call here reaches a kernel or a CUDA API."""
import ctypes
import glob
import math
import os
import re

import pytest
import torch

from fp8_ring_kv_gb300 import kvring as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(K.LIB_PATH):
        from fp8_ring_kv_gb300 import build
        build.build()
    return K.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = re.sub(r"#[^\n]*", " ", text)
        names.update(re.findall(r"\b(kvring_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def paper_config(**kw):
    c = K.make_config(24, 128, 5788, (32, 48, 48), (-40000, 0, 0), (80000, 64, 64))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_header_declares_the_calls():
    names = declared_functions()
    for must in ("kvring_create", "kvring_write", "kvring_reset_positions", "kvring_attend", "kvring_destroy",
                 "kvring_workspace_bytes"):
        assert must in names


def test_every_declared_function_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported by libkvring.so"


def test_binding_uses_the_same_names(lib):
    for name in declared_functions():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name} has no ctypes signature in the binding"


def test_workspace_bytes_valid_configuration(lib):
    c = paper_config()
    n = K.kvring_workspace_bytes(c)
    H, D, S = 24, 128, 5788
    # at least the two code arrays, the two scale arrays and the query scratch
    assert n >= 2 * H * S * D + 2 * H * S * 4 + S * H * D
    assert n % 1024 == 0
    # grows with the ring and with the query scratch
    assert K.kvring_workspace_bytes(paper_config(n_slots=S + 1000)) > n
    assert K.kvring_workspace_bytes(paper_config(max_queries=2 * S)) > n
    assert K.kvring_workspace_bytes(paper_config(max_queries=1)) < n
    # global slots are part of the n_slots, not extra
    assert K.kvring_workspace_bytes(paper_config(n_global=1246)) == n
    assert K.kvring_workspace_bytes(paper_config(n_global=5787)) == n
    assert K.kvring_workspace_bytes(paper_config(scale_mode=K.KVRING_SCALES_STATIC)) == n


@pytest.mark.parametrize("field,value", [
    ("head_dim", 96), ("head_dim", 256), ("heads", 0), ("n_slots", 0), ("n_slots", (1 << 20) + 1),
    ("n_axes", 0), ("n_axes", 4), ("rope_base", 1.0), ("rope_base", math.nan), ("rope_base", math.inf),
    ("out_dtype", 7), ("max_queries", 0), ("max_queries", (1 << 20) + 1),
    ("n_global", -1), ("n_global", 5788), ("n_global", 6000), ("scale_mode", 2), ("scale_mode", -1),
])
def test_workspace_bytes_rejects_invalid(lib, field, value):
    assert K.kvring_workspace_bytes(paper_config(**{field: value})) == 0


def test_head_count_limit(lib):
    """2 * heads * head_dim / 16 <= 1024 (one block of at most 512 threads per
    token in the write and query kernels): 64 heads at D = 128, 128 at D = 64."""
    for heads, dim, ok in ((64, 128, True), (65, 128, False), (128, 64, True), (129, 64, False)):
        c = K.make_config(heads, dim, 512, (dim,), (0,), (1024,))
        assert (K.kvring_workspace_bytes(c) > 0) == ok, (heads, dim)


def test_workspace_bytes_rejects_bad_axes(lib):
    c = paper_config()
    c.axis_dims[0] = 30                       # axes no longer sum to head_dim
    assert K.kvring_workspace_bytes(c) == 0
    c = paper_config()
    c.axis_dims[1], c.axis_dims[2] = 47, 49   # odd axis
    assert K.kvring_workspace_bytes(c) == 0
    c = paper_config()
    c.pos_count[0] = 0
    assert K.kvring_workspace_bytes(c) == 0


def test_status_strings(lib):
    codes = [K.KVRING_OK, K.KVRING_ERR_INVALID_ARG, K.KVRING_ERR_MISALIGNED, K.KVRING_ERR_UNSUPPORTED,
             K.KVRING_ERR_CUDA, K.KVRING_ERR_WORKSPACE, K.KVRING_ERR_NO_DEVICE, K.KVRING_ERR_SCRATCH_LIMIT,
             K.KVRING_ERR_SEQUENCE]
    texts = [lib.kvring_status_string(c).decode() for c in codes]
    assert len(set(texts)) == len(texts) and all(texts)
    assert lib.kvring_status_string(12345).decode() == "unknown status"


def _vp(x):
    return ctypes.c_void_p(x)


def test_create_rejects_before_any_cuda_call(lib):
    c = paper_config()
    need = K.kvring_workspace_bytes(c)
    h = ctypes.c_void_p()
    # the fake workspace addresses are never dereferenced: each case fails a host check first
    assert lib.kvring_create(None, _vp(1 << 20), need, None, ctypes.byref(h)) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_create(ctypes.byref(c), None, need, None, ctypes.byref(h)) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_create(ctypes.byref(c), _vp((1 << 20) + 16), need, None, ctypes.byref(h)) \
        == K.KVRING_ERR_MISALIGNED
    assert lib.kvring_create(ctypes.byref(c), _vp(1 << 20), need - 1, None, ctypes.byref(h)) \
        == K.KVRING_ERR_WORKSPACE
    assert h.value is None
    bad = paper_config(head_dim=96)
    assert lib.kvring_create(ctypes.byref(bad), _vp(1 << 20), need, None, ctypes.byref(h)) \
        == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_create(ctypes.byref(c), _vp(1 << 20), need, None, None) == K.KVRING_ERR_INVALID_ARG


def test_calls_on_null_handle(lib):
    p = _vp(1 << 20)
    assert lib.kvring_write(None, p, p, p, 1, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_write_global(None, p, p, p, 1, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_calibrate(None, 1.5, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_set_qk_norm(None, None, None, 1e-6) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_reset_positions(None, 5, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_attend(None, p, p, 1, p, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_attend_noalloc(None, p, p, 1, p, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_destroy(None) == K.KVRING_OK
    out3 = (ctypes.c_int32 * 3)()
    assert lib.kvring_debug_state(None, None, out3) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_layout(None, None, None, None, None, None, None) == K.KVRING_ERR_INVALID_ARG


def test_debug_quantize_host_checks(lib):
    p = _vp(1 << 20)
    assert lib.kvring_debug_quantize(None, 4, 128, p, p, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_debug_quantize(p, 0, 128, p, p, None) == K.KVRING_ERR_INVALID_ARG
    assert lib.kvring_debug_quantize(p, 4, 48, p, p, None) == K.KVRING_ERR_UNSUPPORTED
    assert lib.kvring_debug_quantize(_vp((1 << 20) + 4), 4, 128, p, p, None) == K.KVRING_ERR_MISALIGNED
    assert lib.kvring_debug_quantize(p, 4, 128, p, _vp((1 << 20) + 2), None) == K.KVRING_ERR_MISALIGNED


def test_binding_constants_match_the_header():
    """Every KVRING_* constant the header defines has the same value in the binding."""
    text = open(HEADERS[0]).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    found = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", text, flags=re.S):
        for name, value in re.findall(r"(KVRING_[A-Z0-9_]+)\s*=\s*(-?\d+)", body):
            found[name] = int(value)
    m = re.search(r"#define\s+KVRING_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    found["KVRING_NOALLOC_SCRATCH_BYTES"] = int(m.group(1)) << int(m.group(2))
    assert len(found) >= 17          # 9 status codes, 3 device error bits, 2 output types, 2 scale modes, 1 size
    for name, value in found.items():
        assert getattr(K, name) == value, name


def test_norm_weights_are_checked_in_the_binding():
    """kvring_set_qk_norm's weights are read as bf16 [H][D] on the device:
    anything else is refused before the library is called."""
    from fp8_ring_kv_gb300 import kvring as K
    with pytest.raises(K.KVRingError, match="bf16"):
        K.kvring_set_qk_norm(None, torch.zeros(4, dtype=torch.float32), None)
    with pytest.raises(K.KVRingError, match="bf16"):
        K.kvring_set_qk_norm(None, None, torch.zeros(4, dtype=torch.bfloat16))   # not on a GPU


def test_ring_wrapper_checks_tensor_arguments():
    """The KVRing wrapper's checks of the token, position and output tensors
    (shape, dtype, contiguity, device) before any call reaches the library."""
    from fp8_ring_kv_gb300.kvring import KVRingError, _check_rows
    cpu = torch.device("cpu")
    k = torch.zeros((5, 3, 64), dtype=torch.bfloat16)
    _check_rows(k, 5, (3, 64), torch.bfloat16, cpu, "k")              # as the kernels read it
    _check_rows(k, 4, (3, 64), torch.bfloat16, cpu, "k")              # extra rows are not read
    for t, n, msg in ((k, 6, "shape"), (k[:, :2], 5, "shape"), (k.float(), 5, "float32"),
                      (torch.zeros((64, 3, 5), dtype=torch.bfloat16).transpose(0, 2), 5, "contiguous")):
        with pytest.raises(KVRingError, match=msg):
            _check_rows(t, n, (3, 64), torch.bfloat16, cpu, "k")
    with pytest.raises(KVRingError, match="the ring is on"):
        _check_rows(k, 5, (3, 64), torch.bfloat16, torch.device("cuda", 0), "k")
    pos = torch.zeros((5, 3), dtype=torch.int64)
    with pytest.raises(KVRingError, match="int64"):
        _check_rows(pos, 5, (3,), torch.int32, cpu, "pos")
