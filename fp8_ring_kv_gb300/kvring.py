"""ctypes binding of libkvring (include/kvring.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory (the workspace and the I/O tensors)
and streams.  The library must be built (``fp8_ring_kv_gb300.build``); if it
is missing, loading fails loudly -- there is no other implementation.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvring.so")

KVRING_OK = 0
KVRING_ERR_INVALID_ARG = -1
KVRING_ERR_MISALIGNED = -2
KVRING_ERR_UNSUPPORTED = -3
KVRING_ERR_CUDA = -4
KVRING_ERR_WORKSPACE = -5
KVRING_ERR_NO_DEVICE = -6
KVRING_ERR_SCRATCH_LIMIT = -7
KVRING_ERR_SEQUENCE = -8
KVRING_NOALLOC_SCRATCH_BYTES = 8 << 20

KVRING_DEVERR_POS_RANGE = 1
KVRING_DEVERR_EMPTY = 2
KVRING_DEVERR_TIMEOUT = 4

KVRING_OUT_BF16 = 0
KVRING_OUT_F32 = 1

KVRING_SCALES_TOKEN = 0
KVRING_SCALES_STATIC = 1

EXPORTS = (
    "kvring_workspace_bytes", "kvring_create", "kvring_write", "kvring_write_global", "kvring_calibrate",
    "kvring_set_qk_norm",
    "kvring_reset_positions", "kvring_reset_positions_batch",
    "kvring_attend", "kvring_destroy", "kvring_status_string", "kvring_last_cuda_error",
    "kvring_layout", "kvring_debug_state", "kvring_debug_quantize", "kvring_attend_noalloc",
    "kvring_debug_wait_timeout",
)


class kvring_config(ctypes.Structure):
    _fields_ = [
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("n_slots", ctypes.c_int32),
        ("n_axes", ctypes.c_int32),
        ("axis_dims", ctypes.c_int32 * 3),
        ("pos_min", ctypes.c_int32 * 3),
        ("pos_count", ctypes.c_int32 * 3),
        ("rope_base", ctypes.c_double),
        ("out_dtype", ctypes.c_int32),
        ("max_queries", ctypes.c_int32),
        ("n_global", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
    ]


class KVRingError(RuntimeError):
    pass


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvring.so (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libkvring is not built ({path} missing): run fp8_ring_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(kvring_config)
    sig = {
        "kvring_workspace_bytes": (sz, [cfgp]),
        "kvring_create": (ctypes.c_int, [cfgp, vp, sz, vp, ctypes.POINTER(vp)]),
        "kvring_write": (ctypes.c_int, [vp, vp, vp, vp, i32, vp]),
        "kvring_write_global": (ctypes.c_int, [vp, vp, vp, vp, i32, vp]),
        "kvring_calibrate": (ctypes.c_int, [vp, ctypes.c_float, vp]),
        "kvring_set_qk_norm": (ctypes.c_int, [vp, vp, vp, ctypes.c_float]),
        "kvring_reset_positions": (ctypes.c_int, [vp, i32, vp]),
        "kvring_reset_positions_batch": (ctypes.c_int, [ctypes.POINTER(vp), i32, i32, vp]),
        "kvring_attend": (ctypes.c_int, [vp, vp, vp, i32, vp, vp]),
        "kvring_attend_noalloc": (ctypes.c_int, [vp, vp, vp, i32, vp, vp]),
        "kvring_destroy": (ctypes.c_int, [vp]),
        "kvring_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kvring_last_cuda_error": (ctypes.c_int, []),
        "kvring_layout": (ctypes.c_int, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                         ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i32)]),
        "kvring_debug_state": (ctypes.c_int, [vp, vp, ctypes.POINTER(i32)]),
        "kvring_debug_quantize": (ctypes.c_int, [vp, i64, i32, vp, vp, vp]),
        "kvring_debug_wait_timeout": (ctypes.c_int, [i64, i32, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, what: str = "") -> None:
    if status != KVRING_OK:
        lib = load()
        msg = lib.kvring_status_string(status).decode()
        if status == KVRING_ERR_CUDA:
            msg += f" (cudaError {lib.kvring_last_cuda_error()})"
        raise KVRingError(f"{what}: {msg} [{status}]")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t if isinstance(t, int) else t.data_ptr())


def make_config(heads, head_dim, n_slots, axis_dims, pos_min, pos_count, rope_base=10000.0,
                out_dtype=KVRING_OUT_F32, max_queries=None, n_global=0,
                scale_mode=KVRING_SCALES_TOKEN) -> kvring_config:
    """max_queries defaults to n_slots (a call attends at most one ring's worth of queries)."""
    c = kvring_config()
    c.heads, c.head_dim, c.n_slots = int(heads), int(head_dim), int(n_slots)
    c.n_axes = len(axis_dims)
    for a in range(3):
        c.axis_dims[a] = int(axis_dims[a]) if a < len(axis_dims) else 0
        c.pos_min[a] = int(pos_min[a]) if a < len(axis_dims) else 0
        c.pos_count[a] = int(pos_count[a]) if a < len(axis_dims) else 0
    c.rope_base = float(rope_base)
    c.out_dtype = int(out_dtype)
    c.max_queries = int(n_slots if max_queries is None else max_queries)
    c.n_global = int(n_global)
    c.scale_mode = int(scale_mode)
    return c


# --- the C-ABI calls under their own names ----------------------------------
def kvring_workspace_bytes(cfg: kvring_config) -> int:
    return int(load().kvring_workspace_bytes(ctypes.byref(cfg)))


def kvring_create(cfg: kvring_config, workspace: torch.Tensor, stream=None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    check(load().kvring_create(ctypes.byref(cfg), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream), ctypes.byref(h)), "kvring_create")
    return h


def kvring_write(handle, k, v, pos, n_new: int, stream=None) -> None:
    check(load().kvring_write(handle, _ptr(k), _ptr(v), _ptr(pos), int(n_new), _stream(stream)), "kvring_write")


def kvring_write_global(handle, k, v, pos, n: int, stream=None) -> None:
    check(load().kvring_write_global(handle, _ptr(k), _ptr(v), _ptr(pos), int(n), _stream(stream)),
          "kvring_write_global")


def _check_rows(t, n, trailing, dtype, device, what):
    """A tensor the kernels read or write as n rows of ``trailing`` elements:
    at least n rows (the kernels touch the first n only), of ``dtype``,
    contiguous, on the ring's ``device``."""
    shape = t.shape
    if shape[1:] != trailing or shape[0] < n:
        raise KVRingError(f"{what}: shape {tuple(shape)}; the call reads [{n}, {', '.join(map(str, trailing))}]")
    if t.dtype != dtype:
        raise KVRingError(f"{what}: {t.dtype}; the kernels read {dtype}")
    if not t.is_contiguous():
        raise KVRingError(f"{what}: not contiguous")
    if t.device != device:
        raise KVRingError(f"{what}: on {t.device}, the ring is on {device}")


def _check_norm_weight(w, numel, device, what):
    """A norm weight as the kernels read it: contiguous bf16 on the ring's
    device with exactly H * D values."""
    if w is None or isinstance(w, int):
        return
    if w.dtype != torch.bfloat16 or not w.is_cuda or not w.is_contiguous():
        raise KVRingError(f"{what}: a contiguous bf16 CUDA tensor is required")
    if numel is not None and w.numel() != numel:
        raise KVRingError(f"{what}: {w.numel()} values, the ring needs H * D = {numel} "
                          "(expand a weight shared by all heads to [H, D])")
    if device is not None and w.device != torch.device(device):
        raise KVRingError(f"{what}: on {w.device}, the ring is on {device}")


def kvring_set_qk_norm(handle, gamma_q=None, gamma_k=None, eps: float = 1e-6, numel=None, device=None) -> None:
    """gamma_q / gamma_k: bf16 [H, D] CUDA tensors (or raw device addresses,
    unchecked); numel / device, when given, are checked against the tensors."""
    _check_norm_weight(gamma_q, numel, device, "kvring_set_qk_norm gamma_q")
    _check_norm_weight(gamma_k, numel, device, "kvring_set_qk_norm gamma_k")
    gq = None if gamma_q is None else _ptr(gamma_q)
    gk = None if gamma_k is None else _ptr(gamma_k)
    check(load().kvring_set_qk_norm(handle, gq, gk, float(eps)), "kvring_set_qk_norm")


def kvring_calibrate(handle, margin: float = 1.5, stream=None) -> None:
    check(load().kvring_calibrate(handle, float(margin), _stream(stream)), "kvring_calibrate")


def kvring_reset_positions(handle, d: int, stream=None) -> None:
    check(load().kvring_reset_positions(handle, int(d), _stream(stream)), "kvring_reset_positions")


def kvring_reset_positions_batch(handles, d: int, stream=None) -> None:
    arr = (ctypes.c_void_p * len(handles))(*[h.value if isinstance(h, ctypes.c_void_p) else h for h in handles])
    check(load().kvring_reset_positions_batch(arr, len(handles), int(d), _stream(stream)),
          "kvring_reset_positions_batch")


def kvring_attend(handle, q, q_pos, n_q: int, out, stream=None) -> None:
    check(load().kvring_attend(handle, _ptr(q), _ptr(q_pos), int(n_q), _ptr(out), _stream(stream)),
          "kvring_attend")


def kvring_attend_noalloc(handle, q, q_pos, n_q: int, out, stream=None) -> None:
    """kvring_attend with the query scratch in the library's fixed device array
    (no allocation; concurrent calls on one device race on that array)."""
    check(load().kvring_attend_noalloc(handle, _ptr(q), _ptr(q_pos), int(n_q), _ptr(out), _stream(stream)),
          "kvring_attend_noalloc")


def kvring_destroy(handle) -> None:
    check(load().kvring_destroy(handle), "kvring_destroy")


def kvring_debug_wait_timeout(limit_ns: int, complete: bool, out2, stream=None) -> None:
    """The library's bounded barrier wait on its own (see kvring.h); out2: int64 [2] CUDA tensor."""
    check(load().kvring_debug_wait_timeout(int(limit_ns), int(bool(complete)), _ptr(out2), _stream(stream)),
          "kvring_debug_wait_timeout")


def kvring_debug_quantize(x, rows: int, d: int, codes, scales, stream=None) -> None:
    check(load().kvring_debug_quantize(_ptr(x), int(rows), int(d), _ptr(codes), _ptr(scales), _stream(stream)),
          "kvring_debug_quantize")


# --- a convenience object over one ring ----------------------------------------
class KVRing:
    """One ring in a torch-allocated device workspace.

    ``write``/``reset_positions``/``attend`` enqueue the library's kernels on
    the current (or given) stream and return at once."""

    def __init__(self, heads, head_dim, n_slots, axis_dims, pos_min, pos_count, rope_base=10000.0,
                 out_dtype=KVRING_OUT_F32, device="cuda", stream=None, max_queries=None, n_global=0,
                 scale_mode=KVRING_SCALES_TOKEN, workspace=None):
        self.cfg = make_config(heads, head_dim, n_slots, axis_dims, pos_min, pos_count, rope_base, out_dtype,
                               max_queries, n_global, scale_mode)
        nbytes = kvring_workspace_bytes(self.cfg)
        if nbytes == 0:
            raise KVRingError("invalid kvring configuration")
        self.heads, self.head_dim, self.n_slots = int(heads), int(head_dim), int(n_slots)
        self.n_global = int(n_global)
        self.n_axes = len(axis_dims)
        self.out_dtype = torch.float32 if out_dtype == KVRING_OUT_F32 else torch.bfloat16
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        elif workspace.dtype != torch.uint8 or workspace.numel() < nbytes or workspace.data_ptr() % 256:
            raise KVRingError("workspace: a uint8 tensor of kvring_workspace_bytes, 256-byte aligned")
        self.workspace = workspace
        self.handle = kvring_create(self.cfg, self.workspace, stream)
        ptrs = [ctypes.c_void_p() for _ in range(5)]
        s_pad = ctypes.c_int32()
        check(load().kvring_layout(self.handle, *[ctypes.byref(p) for p in ptrs], ctypes.byref(s_pad)),
              "kvring_layout")
        self.s_pad = int(s_pad.value)
        base = self.workspace.data_ptr()
        off = [p.value - base for p in ptrs]
        H, S, D = self.heads, self.n_slots, self.head_dim
        ws = self.workspace
        self.k_codes = ws[off[0]:off[0] + H * S * D].view(H, S, D)
        self.v_codes = ws[off[1]:off[1] + H * S * D].view(H, S, D)
        self.k_scales = ws[off[2]:off[2] + H * self.s_pad * 4].view(torch.float32).view(H, self.s_pad)
        self.v_scales = ws[off[3]:off[3] + H * self.s_pad * 4].view(torch.float32).view(H, self.s_pad)
        self.state_words = ws[off[4]:off[4] + 16].view(torch.int32)

    @classmethod
    def from_shape(cls, shape, out_dtype=KVRING_OUT_F32, device="cuda", stream=None, max_queries=None,
                   workspace=None):
        return cls(shape.heads, shape.head_dim, shape.n_slots, shape.axis_dims, shape.pos_min, shape.pos_count,
                   shape.rope_base, out_dtype, device, stream, max_queries, getattr(shape, "n_global", 0),
                   KVRING_SCALES_STATIC if getattr(shape, "scale_mode", "token") == "static" else KVRING_SCALES_TOKEN,
                   workspace)

    def _check_tokens(self, what, n, pairs):
        """bf16 [n, H, D] token tensors and int32 [n, n_axes] positions on the ring's device."""
        dev = self.workspace.device
        for name, t in pairs:
            if name.endswith("pos"):
                _check_rows(t, n, (self.n_axes,), torch.int32, dev, name)
            else:
                _check_rows(t, n, (self.heads, self.head_dim), torch.bfloat16, dev, name)

    def write(self, k, v, pos, stream=None):
        n = k.shape[0]
        self._check_tokens("write", n, (("k", k), ("v", v), ("pos", pos)))
        kvring_write(self.handle, k, v, pos, n, stream)

    def write_global(self, k, v, pos, stream=None):
        n = k.shape[0]
        self._check_tokens("write_global", n, (("k", k), ("v", v), ("pos", pos)))
        kvring_write_global(self.handle, k, v, pos, n, stream)

    def calibrate(self, margin=1.5, stream=None):
        kvring_calibrate(self.handle, margin, stream)

    def set_qk_norm(self, gamma_q=None, gamma_k=None, eps=1e-6):
        """bf16 [H, D] device weights (None: off); the tensors are kept alive here."""
        kvring_set_qk_norm(self.handle, gamma_q, gamma_k, eps, numel=self.heads * self.head_dim,
                           device=self.workspace.device)
        self._norm_weights = (gamma_q, gamma_k)

    def reset_positions(self, d, stream=None):
        kvring_reset_positions(self.handle, d, stream)

    def attend(self, q, q_pos, out=None, stream=None):
        n = q.shape[0]
        self._check_tokens("attend", n, (("q", q), ("q_pos", q_pos)))
        if out is None:
            out = torch.empty(q.shape, dtype=self.out_dtype, device=q.device)
        _check_rows(out, n, (self.heads, self.head_dim), self.out_dtype, self.workspace.device, "out")
        kvring_attend(self.handle, q, q_pos, n, out, stream)
        return out

    def debug_state(self, stream=None):
        arr = (ctypes.c_int32 * 3)()
        check(load().kvring_debug_state(self.handle, _stream(stream), arr), "kvring_debug_state")
        return int(arr[0]), int(arr[1]), int(arr[2])

    def close(self):
        if self.handle is not None:
            kvring_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVRingStack:
    """n rings of one shape in ONE device allocation (one slice per ring,
    each ring with its own state), reset together by one batched launch.

    ``rings[i]`` is a KVRing whose workspace is a view of ``self.workspace``."""

    def __init__(self, n, shape, out_dtype=KVRING_OUT_F32, device="cuda", max_queries=None):
        if n < 1:
            raise KVRingError("a stack holds at least one ring")
        cfg = make_config(shape.heads, shape.head_dim, shape.n_slots, shape.axis_dims, shape.pos_min,
                          shape.pos_count, shape.rope_base, out_dtype, max_queries, getattr(shape, "n_global", 0),
                          KVRING_SCALES_STATIC if getattr(shape, "scale_mode", "token") == "static"
                          else KVRING_SCALES_TOKEN)
        stride = kvring_workspace_bytes(cfg)
        if stride == 0:
            raise KVRingError("invalid kvring configuration")
        self.stride = stride
        self.workspace = torch.empty(n * stride, dtype=torch.uint8, device=device)
        self.rings = [KVRing.from_shape(shape, out_dtype, device, max_queries=max_queries,
                                        workspace=self.workspace[i * stride:(i + 1) * stride]) for i in range(n)]

    def reset_positions(self, d, stream=None):
        kvring_reset_positions_batch([r.handle for r in self.rings], d, stream)

    def close(self):
        for r in self.rings:
            r.close()
