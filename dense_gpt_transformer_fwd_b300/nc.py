"""ctypes binding of the nc C ABI (``include/nc.h``).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libnc.so``.  PyTorch provides device memory and streams.  There
is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnc.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "nc.h")

NC_F32, NC_BF16, NC_FP8 = 0, 1, 2
DTYPES = {"f32": NC_F32, "bf16": NC_BF16, "fp8": NC_FP8}
KCLASSES = ("embed", "qkv", "attn", "oproj", "norm", "fc", "proj", "lm_head")
STATUS = {0: "NC_OK", 1: "NC_ERR_INVALID_ARG", 2: "NC_ERR_UNSUPPORTED", 3: "NC_ERR_OOM",
          4: "NC_ERR_STATE", 5: "NC_ERR_CAPACITY", 6: "NC_ERR_TOKEN", 7: "NC_ERR_TIMEOUT",
          8: "NC_ERR_CUDA", 9: "NC_ERR_SCRATCH_LIMIT"}


class NcError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{what}: {self.name}" + (f" ({detail})" if detail else ""))


class NcConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layer", "d_model", "n_head", "n_kv_head", "head_dim", "d_mlp", "vocab")] + \
               [(n, ctypes.c_float) for n in ("rope_base", "softcap", "rms_eps")] + \
               [(n, ctypes.c_int32) for n in ("dtype", "max_batch", "max_seq", "window", "reserved")] + \
               [("window_layers", ctypes.c_uint64)] + \
               [(n, ctypes.c_int32) for n in ("extras", "ve_gate_channels", "smear_channels", "reserved2")]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions declared in include/nc.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:NC_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(nc_[a-z0-9_]+)\s*\(",
                                 text, re.M)))


def lib() -> ctypes.CDLL:
    """Load libnc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m dense_gpt_transformer_fwd_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    sig = {
        "nc_model_create": ([ctypes.POINTER(NcConfig), P, ctypes.POINTER(P)], S),
        "nc_model_destroy": ([P], None),
        "nc_kv_reset": ([P, P], S),
        "nc_prefill": ([P, P, I32, I32, P, I32, P], S),
        "nc_decode_step": ([P, P, I32, P, P], S),
        "nc_prefill_rows": ([P, P, I32, I32, P, P, I32, P], S),
        "nc_kv_row_lengths": ([P, P], S),
        "nc_decode_step_noalloc": ([P, P, I32, P, P], S),
        "nc_sync_status": ([P, P], S),
        "nc_kv_clone": ([P, I32, I32, P], S),
        "nc_sample": ([P, P, I32, ctypes.c_double, I32, P, P, P], S),
        "nc_kv_length": ([P, ctypes.POINTER(I32), ctypes.POINTER(I32)], S),
        "nc_kv_layout": ([P, ctypes.POINTER(I64), ctypes.POINTER(I64), ctypes.POINTER(I32)], S),
        "nc_kv_read": ([P, P, P, P], S),
        "nc_launch_count": ([P], I64),
        "nc_gemm_bf16": ([P, P, P, P, I32, I32, I32, P], S),
        "nc_debug_wait_timeout": ([P, I64, P], S),
        "nc_set_wait_limit": ([P, I64], S),
        "nc_profile_begin": ([P], S),
        "nc_profile_end": ([P, P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)], S),
        "nc_status_string": ([S], ctypes.c_char_p),
        "nc_last_cuda_error": ([], ctypes.c_char_p),
    }
    for name, (argt, rest) in sig.items():
        f = getattr(L, name)
        f.argtypes = argt
        f.restype = rest
    _lib = L
    return L


def _check(code: int, what: str):
    if code != 0:
        detail = ""
        if STATUS.get(code) in ("NC_ERR_CUDA", "NC_ERR_OOM") and _lib is not None:
            detail = _lib.nc_last_cuda_error().decode()
        raise NcError(code, what, detail)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    import torch
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return ctypes.c_void_p(t.data_ptr())
    if isinstance(t, np.ndarray):
        if not t.flags.c_contiguous:
            raise ValueError("array must be C-contiguous")
        return ctypes.c_void_p(t.ctypes.data)
    raise TypeError(type(t))


def window_layers(pattern: str, n_layer: int) -> int:
    """Bit l set where the sliding-window pattern (e.g. "SSSL", repeated over
    the layers) has an "S" at layer l."""
    if not pattern:
        return 0
    return sum(1 << l for l in range(n_layer) if pattern[l % len(pattern)] == "S")


def make_config(shape, max_batch: int, max_seq: int) -> NcConfig:
    """nc_config from a shape object with the nc_inputs.ModelShape fields."""
    window = int(getattr(shape, "window", 0) or 0)
    pattern = getattr(shape, "window_pattern", "") or ""
    extras = sum(bit for bit, flag in ((1, "value_embeds"), (2, "resid_lambdas"), (4, "smear"), (8, "backout"))
                 if getattr(shape, flag, False))
    return NcConfig(shape.n_layer, shape.d_model, shape.n_head, shape.n_kv_head, shape.head_dim,
                    shape.d_mlp, shape.vocab, shape.rope_base, shape.softcap, shape.rms_eps,
                    DTYPES[shape.dtype], max_batch, max_seq,
                    window if pattern else 0, 0, window_layers(pattern, shape.n_layer) if window else 0,
                    extras, int(getattr(shape, "ve_gate_channels", 32)), int(getattr(shape, "smear_channels", 24)),
                    0)


class Model:
    """A model on the current CUDA device (see nc_model_create).

    ``weights``: packed fp32 vector in canonical order (numpy array or torch
    tensor, host or device).  ``prefill``/``decode_step`` take int32 tokens as
    torch tensors (device or host) and return fp32 logits on the same side.
    """

    def __init__(self, shape, weights, max_batch: int, max_seq: int, cfg: NcConfig | None = None):
        self._L = lib()
        self.shape = shape
        self.cfg = cfg if cfg is not None else make_config(shape, max_batch, max_seq)
        self._h = ctypes.c_void_p()
        w = weights
        if isinstance(w, np.ndarray):
            w = np.ascontiguousarray(w, dtype=np.float32)
        _check(self._L.nc_model_create(ctypes.byref(self.cfg), _ptr(w), ctypes.byref(self._h)),
               "nc_model_create")

    def close(self):
        if self._h:
            self._L.nc_model_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def _out(self, tokens, rows):
        import torch
        V = self.cfg.vocab
        if tokens.is_cuda:
            return torch.empty((rows, V), dtype=torch.float32, device=tokens.device)
        return torch.empty((rows, V), dtype=torch.float32, pin_memory=True)

    def prefill(self, tokens, last_only: bool = False, out=None, stream=None):
        import torch
        tokens = tokens.to(torch.int32).contiguous() if tokens.dtype != torch.int32 else tokens.contiguous()
        B, T = tokens.shape
        if out is None:
            out = self._out(tokens, B if last_only else B * T)
        _check(self._L.nc_prefill(self._h, _ptr(tokens), B, T, _ptr(out), int(last_only),
                                  _stream(stream)), "nc_prefill")
        return out.view(B, self.cfg.vocab) if last_only else out.view(B, T, self.cfg.vocab)

    def prefill_rows(self, tokens, row_len, last_only: bool = False, out=None, stream=None):
        """nc_prefill_rows: tokens [B, T] with row_len[b] real tokens at the
        start of row b (host int sequence); each row keeps its own length."""
        import torch
        tokens = tokens.to(torch.int32).contiguous()
        B, T = tokens.shape
        lens = np.ascontiguousarray(np.asarray(row_len, dtype=np.int32).reshape(B))
        if out is None:
            out = self._out(tokens, B if last_only else B * T)
        _check(self._L.nc_prefill_rows(self._h, _ptr(tokens), B, T, _ptr(lens), _ptr(out), int(last_only),
                                       _stream(stream)), "nc_prefill_rows")
        return out.view(B, self.cfg.vocab) if last_only else out.view(B, T, self.cfg.vocab)

    def row_lengths(self):
        """Each cached row's length (host list)."""
        n, b = self.kv_length()
        out = np.zeros(max(b, 1), dtype=np.int32)
        _check(self._L.nc_kv_row_lengths(self._h, _ptr(out)), "nc_kv_row_lengths")
        return out[:b].tolist()

    def decode_step(self, tokens, out=None, stream=None):
        import torch
        tokens = tokens.to(torch.int32).contiguous()
        B = tokens.numel()
        if out is None:
            out = self._out(tokens, B)
        _check(self._L.nc_decode_step(self._h, _ptr(tokens), B, _ptr(out), _stream(stream)),
               "nc_decode_step")
        return out.view(B, self.cfg.vocab)

    def decode_step_noalloc(self, tokens, out, stream=None):
        """nc_decode_step_noalloc: device tokens [B] int32 and a caller-owned
        device logits buffer [B, V] fp32; allocates nothing."""
        B = tokens.numel()
        _check(self._L.nc_decode_step_noalloc(self._h, _ptr(tokens), B, _ptr(out), _stream(stream)),
               "nc_decode_step_noalloc")
        return out.view(B, self.cfg.vocab)

    def kv_clone(self, src: int, n: int, stream=None):
        """nc_kv_clone: rows [0, n) of the cache become copies of row src."""
        _check(self._L.nc_kv_clone(self._h, int(src), int(n), _stream(stream)), "nc_kv_clone")

    def sample(self, logits, temperature: float = 0.0, top_k: int = 0, u=None, out=None, stream=None):
        """nc_sample: next tokens [B] int32 (device) from device logits [B, V]
        fp32; u: device fp64 draws [B] (needed when temperature > 0)."""
        import torch
        B = logits.shape[0]
        if out is None:
            out = torch.empty(B, dtype=torch.int32, device=logits.device)
        up = _ptr(u) if u is not None else ctypes.c_void_p()
        _check(self._L.nc_sample(self._h, _ptr(logits), B, float(temperature), int(top_k), up, _ptr(out),
                                 _stream(stream)), "nc_sample")
        return out

    def kv_reset(self, stream=None):
        _check(self._L.nc_kv_reset(self._h, _stream(stream)), "nc_kv_reset")

    def sync(self, stream=None):
        """Synchronize and raise NcError on a recorded device error."""
        _check(self._L.nc_sync_status(self._h, _stream(stream)), "nc_sync_status")

    def sync_status(self, stream=None) -> int:
        return self._L.nc_sync_status(self._h, _stream(stream))

    def kv_length(self):
        n, b = ctypes.c_int32(), ctypes.c_int32()
        _check(self._L.nc_kv_length(self._h, ctypes.byref(n), ctypes.byref(b)), "nc_kv_length")
        return n.value, b.value

    def kv_read(self):
        """Raw K and V caches with guards: (k, v, guard_elems, elem_bytes), on the device."""
        import torch
        total, guard, eb = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _check(self._L.nc_kv_layout(self._h, ctypes.byref(total), ctypes.byref(guard),
                                    ctypes.byref(eb)), "nc_kv_layout")
        dt = torch.int16 if eb.value == 2 else torch.int32
        n = total.value // eb.value
        k = torch.empty(n, dtype=dt, device="cuda")
        v = torch.empty(n, dtype=dt, device="cuda")
        _check(self._L.nc_kv_read(self._h, _ptr(k), _ptr(v), _stream(None)), "nc_kv_read")
        torch.cuda.current_stream().synchronize()
        return k, v, guard.value, eb.value

    @property
    def launch_count(self) -> int:
        return int(self._L.nc_launch_count(self._h))

    def gemm_bf16(self, A, W, C, stream=None):
        M, K = A.shape
        N = W.shape[0]
        _check(self._L.nc_gemm_bf16(self._h, _ptr(A), _ptr(W), _ptr(C), M, N, K, _stream(stream)),
               "nc_gemm_bf16")
        return C

    def debug_wait_timeout(self, limit_ns: int, stream=None):
        _check(self._L.nc_debug_wait_timeout(self._h, int(limit_ns), _stream(stream)),
               "nc_debug_wait_timeout")

    def set_wait_limit(self, limit_ns: int):
        _check(self._L.nc_set_wait_limit(self._h, int(limit_ns)), "nc_set_wait_limit")

    def profile_begin(self):
        _check(self._L.nc_profile_begin(self._h), "nc_profile_begin")

    def profile_end(self, stream=None) -> dict:
        """Per kernel class: (device ms summed over launches, launches)."""
        n = len(KCLASSES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        _check(self._L.nc_profile_end(self._h, _stream(stream), ms, cnt), "nc_profile_end")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(KCLASSES)}
