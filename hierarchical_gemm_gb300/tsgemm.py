"""Python binding of the tsgemm C ABI (ctypes).

Argument marshalling only: every step of C = A * B runs in the CUDA kernels
of libtsgemm.so.  There is no fallback path; if the library has not been
built, importing this module raises ImportError.
"""
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libtsgemm.so")

F16, BF16, F32 = 0, 1, 2
E4M3, E5M2 = 3, 4  # 8-bit float inputs (OCP FP8), RCR layout only
# operand storage: A M x K or K x M (column-major), B K x N or N x K
LAYOUT_RRR, LAYOUT_RCR, LAYOUT_CRR, LAYOUT_CCR = 0, 1, 2, 3
_LAYOUT_NAMES = {"rrr": LAYOUT_RRR, "rcr": LAYOUT_RCR, "crr": LAYOUT_CRR, "ccr": LAYOUT_CCR}

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_ALIGNMENT = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_OOM = 6
ERR_SCRATCH_LIMIT = 7

DEBUG_SKIP_FIRST_LOAD = 1

_DTYPE_NAMES = {"f16": F16, "fp16": F16, "float16": F16, "half": F16,
                "bf16": BF16, "bfloat16": BF16,
                "f32": F32, "fp32": F32, "float32": F32, "float": F32,
                "e4m3": E4M3, "float8_e4m3fn": E4M3, "e5m2": E5M2, "float8_e5m2": E5M2}

# Every entry point include/tsgemm.h and include/tsattn.h declare.
EXPORTS = ("tsgemm_plan", "tsgemm_plan_ex", "tsgemm_run", "tsgemm_destroy",
           "tsgemm_status", "tsgemm_get_config", "tsgemm_choose_config",
           "tsgemm_status_string", "tsgemm_run_splitk_noalloc",
           "tsattn_forward", "tsattn_forward_ex", "tsattn_mla_decode", "tsattn_mla_decode_ex",
           "tsattn_status")


class Config(ctypes.Structure):
    """Mirror of tsgemm_config_t."""
    _fields_ = [("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("units", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("timeout_ms", ctypes.c_int32), ("debug_flags", ctypes.c_int32),
                ("split_tiles", ctypes.c_int64), ("stream_k_tiles", ctypes.c_int64),
                ("cluster_split", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libtsgemm.so is not built (%s); run hierarchical_gemm_gb300.build.build() "
            "or __graft_entry__.build() first" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    cfgp = ctypes.POINTER(Config)
    L.tsgemm_plan.restype = i32
    L.tsgemm_plan.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32]
    L.tsgemm_plan_ex.restype = i32
    L.tsgemm_plan_ex.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32, cfgp]
    L.tsgemm_run.restype = i32
    L.tsgemm_run.argtypes = [vp, vp, vp, vp, vp]
    L.tsgemm_destroy.restype = i32
    L.tsgemm_destroy.argtypes = [vp]
    L.tsgemm_status.restype = i32
    L.tsgemm_status.argtypes = [vp]
    L.tsgemm_get_config.restype = i32
    L.tsgemm_get_config.argtypes = [vp, cfgp]
    L.tsgemm_choose_config.restype = i32
    L.tsgemm_choose_config.argtypes = [i64, i64, i64, i32, i32, i32, i32, cfgp, cfgp]
    L.tsgemm_status_string.restype = ctypes.c_char_p
    L.tsgemm_status_string.argtypes = [i32]
    L.tsgemm_run_splitk_noalloc.restype = i32
    L.tsgemm_run_splitk_noalloc.argtypes = [i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp]
    f32 = ctypes.c_float
    L.tsattn_forward.restype = i32
    L.tsattn_forward.argtypes = [i64, i64, i64, i64, i32, i32, f32, i32, vp, vp, vp, vp, vp, vp]
    L.tsattn_forward_ex.restype = i32
    L.tsattn_forward_ex.argtypes = [i64, i64, i64, i64, i32, i32, f32, i32, vp, vp, vp, vp, vp, vp, i32, i32]
    L.tsattn_mla_decode.restype = i32
    L.tsattn_mla_decode.argtypes = [i64, i64, i64, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, vp]
    L.tsattn_mla_decode_ex.restype = i32
    L.tsattn_mla_decode_ex.argtypes = [i64, i64, i64, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32]
    L.tsattn_status.restype = i32
    L.tsattn_status.argtypes = []
    return L


lib = _load()


class TsgemmError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


def status_string(code):
    return lib.tsgemm_status_string(int(code)).decode()


def _check(code, what):
    if code != OK:
        raise TsgemmError(code, what)


def dtype_code(d):
    """tsgemm dtype code from a name, a code or a torch dtype."""
    if isinstance(d, int):
        return d
    s = str(d).lower().replace("torch.", "")
    return _DTYPE_NAMES[s]


def layout_code(layout):
    """tsgemm layout code from a code or a name ("rrr", "rcr", "crr", "ccr")."""
    if isinstance(layout, int):
        return layout
    return _LAYOUT_NAMES[str(layout).lower()]


def _force(kw):
    c = Config()
    for k, v in kw.items():
        if not hasattr(c, k):
            raise TypeError("unknown configuration field %r" % k)
        setattr(c, k, int(v))
    return c


def choose_config(M, N, K, dtype_in, dtype_out, num_sms, layout=LAYOUT_RRR, **force):
    """The planner's configuration for a problem (host only, no GPU)."""
    out = Config()
    f = _force(force)
    _check(lib.tsgemm_choose_config(M, N, K, dtype_code(dtype_in), dtype_code(dtype_out),
                                    layout_code(layout), int(num_sms), ctypes.byref(f), ctypes.byref(out)),
           "tsgemm_choose_config")
    return out.as_dict()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """A planned GEMM C (M x N) = A (M x K) * B (K x N) on the current device.

    `layout` says how A and B are stored (LAYOUT_RRR: A M x K and B K x N
    row-major; RCR: B stored N x K; CRR: A stored K x M; CCR: both)."""

    def __init__(self, M, N, K, dtype_in, dtype_out, layout=LAYOUT_RRR, **force):
        self._h = ctypes.c_void_p()
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.dtype_in, self.dtype_out = dtype_code(dtype_in), dtype_code(dtype_out)
        self.layout = layout_code(layout)
        if force:
            f = _force(force)
            code = lib.tsgemm_plan_ex(ctypes.byref(self._h), self.M, self.N, self.K,
                                      self.dtype_in, self.dtype_out, self.layout, ctypes.byref(f))
        else:
            code = lib.tsgemm_plan(ctypes.byref(self._h), self.M, self.N, self.K,
                                   self.dtype_in, self.dtype_out, self.layout)
        _check(code, "tsgemm_plan")

    @property
    def config(self):
        out = Config()
        _check(lib.tsgemm_get_config(self._h, ctypes.byref(out)), "tsgemm_get_config")
        return out.as_dict()

    def run(self, A, B, C, stream=None):
        """Enqueue C = A * B; A, B, C are CUDA tensors (or raw device pointers)."""
        _check(lib.tsgemm_run(self._h, _ptr(A), _ptr(B), _ptr(C), _stream_handle(stream)),
               "tsgemm_run")
        return C

    def status(self):
        """Device status word after the runs have completed (0 = OK)."""
        return lib.tsgemm_status(self._h)

    def close(self):
        if self._h:
            lib.tsgemm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_TORCH_OUT = {F16: "float16", BF16: "bfloat16", F32: "float32"}
_plans = {}


def _storage(X):
    """(column-major?, tensor whose data pointer is the stored matrix) for a
    2-D CUDA tensor that is row-major contiguous or the transpose of one."""
    if X.is_contiguous():
        return False, X
    if X.t().is_contiguous():
        return True, X.t()
    raise ValueError("operands must be row-major contiguous or transposes of contiguous tensors")


def gemm(A, B, out_dtype=None, C=None, stream=None):
    """C = A @ B for CUDA tensors A (M x K) and B (K x N) of dtype float16,
    bfloat16, float8_e4m3fn or float8_e5m2.  Each operand may be row-major
    contiguous or a transposed view of a contiguous tensor (for example
    W.t() of a weight W stored N x K); the layout follows from the strides.
    Plans are cached per shape, dtype and layout."""
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("expected A (M x K) and B (K x N)")
    if A.dtype != B.dtype:
        raise ValueError("A and B must have the same dtype")
    a_col, A_store = _storage(A)
    b_col, B_store = _storage(B)
    layout = (LAYOUT_CRR if a_col else 0) | (LAYOUT_RCR if b_col else 0)
    din = dtype_code(A.dtype)
    dout = dtype_code(out_dtype) if out_dtype is not None else (F32 if C is None else dtype_code(C.dtype))
    M, K = A.shape
    N = B.shape[1]
    key = (A.device.index, M, N, K, din, dout, layout)
    plan = _plans.get(key)
    if plan is None:
        plan = _plans[key] = Plan(M, N, K, din, dout, layout=layout)
    if C is None:
        C = torch.empty((M, N), dtype=getattr(torch, _TORCH_OUT[dout]), device=A.device)
    return plan.run(A_store, B_store, C, stream)


def run_splitk_noalloc(A, B, C, splits=0, status=None, stream=None):
    """C = A * B through the entry point that allocates nothing (its split-K
    scratch is a fixed device array inside the library).  A (M x K), B
    (K x N), C (M x N) are CUDA tensors or raw device pointers; `status` an
    optional device int tensor that receives a device-side timeout."""
    M, K = A.shape
    N = B.shape[1]
    din = dtype_code(A.dtype)
    dout = dtype_code(C.dtype)
    _check(lib.tsgemm_run_splitk_noalloc(M, N, K, din, dout, int(splits), _ptr(A), _ptr(B),
                                         _ptr(C), _ptr(status), _stream_handle(stream)),
           "tsgemm_run_splitk_noalloc")
    return C


def attention(Q, K, V, scale=None, causal=False, O=None, status=None, stream=None, debug_flags=0,
              timeout_ms=0):
    """O = softmax(scale * Q K^T) V for CUDA tensors Q (B, H, Sq, D), K and V
    (B, H, Sk, D), contiguous, all float16 or all bfloat16, D = 128 (the
    attention block of tsattn.h).  scale defaults to D ** -0.5; `causal`
    lets query row i see keys t <= i + Sk - Sq.  `status`: an optional
    device int tensor that receives a device-side timeout."""
    import torch
    if Q.dim() != 4 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("expected Q, K, V of shape (B, H, S, D)")
    B, H, Sq, D = Q.shape
    Sk = K.shape[2]
    if K.shape != (B, H, Sk, D) or V.shape != (B, H, Sk, D):
        raise ValueError("K and V must be (B, H, Sk, D) with Q's B, H and D")
    if not (Q.dtype == K.dtype == V.dtype) or not all(x.is_contiguous() for x in (Q, K, V)):
        raise ValueError("Q, K, V must share a dtype and be contiguous")
    if scale is None:
        scale = float(D) ** -0.5
    if O is None:
        O = torch.empty_like(Q)
    _check(lib.tsattn_forward_ex(B, H, Sq, Sk, D, dtype_code(Q.dtype), float(scale), int(bool(causal)),
                                 _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(status), _stream_handle(stream),
                                 int(debug_flags), int(timeout_ms)),
           "tsattn_forward")
    return O


def mla_decode(Q, Q_pe, KV, K_pe, scale=None, O=None, status=None, stream=None, debug_flags=0, timeout_ms=0,
               prefetch_blocks=0):
    """MLA decode (tsattn_mla_decode): for CUDA tensors Q (B, H, 512), Q_pe
    (B, H, 64), KV (B, Skv, 512) and K_pe (B, Skv, 64), contiguous, all
    float16 or all bfloat16, O (B, H, 512) = softmax(scale * (Q KV^T +
    Q_pe K_pe^T)) KV per batch.  scale defaults to 576 ** -0.5."""
    import torch
    if Q.dim() != 3 or Q_pe.dim() != 3 or KV.dim() != 3 or K_pe.dim() != 3:
        raise ValueError("expected Q (B, H, 512), Q_pe (B, H, 64), KV (B, Skv, 512), K_pe (B, Skv, 64)")
    B, H, dim = Q.shape
    pe_dim = Q_pe.shape[2]
    Skv = KV.shape[1]
    if Q_pe.shape[:2] != (B, H) or KV.shape != (B, Skv, dim) or K_pe.shape != (B, Skv, pe_dim):
        raise ValueError("inconsistent MLA shapes")
    if not (Q.dtype == Q_pe.dtype == KV.dtype == K_pe.dtype) or \
            not all(x.is_contiguous() for x in (Q, Q_pe, KV, K_pe)):
        raise ValueError("Q, Q_pe, KV, K_pe must share a dtype and be contiguous")
    if scale is None:
        scale = float(dim + pe_dim) ** -0.5
    if O is None:
        O = torch.empty_like(Q)
    _check(lib.tsattn_mla_decode_ex(B, H, Skv, dim, pe_dim, dtype_code(Q.dtype), float(scale), _ptr(Q), _ptr(Q_pe),
                                    _ptr(KV), _ptr(K_pe), _ptr(O), _ptr(status), _stream_handle(stream),
                                    int(debug_flags), int(timeout_ms), int(prefetch_blocks)),
           "tsattn_mla_decode")
    return O


def attention_status():
    """The library's own attention status word (0 = OK); reading clears it."""
    return lib.tsattn_status()
