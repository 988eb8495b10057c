"""H2O (Heavy-Hitter Oracle) KV-cache eviction on GB300: Python binding.

A thin ctypes layer over ``libh2o.so`` (C ABI in ``include/h2o.h``).  PyTorch
supplies device memory and the current CUDA stream; every step of prefill and
decode runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or the device is not a CUDA device, calls raise.

    cache = H2OCache(B, H, d, k_heavy, k_local, dtype=torch.bfloat16)
    O, lse, colsum = cache.prefill(Q, K, V)          # [B,H,L,d] each
    out = cache.step(q_t, k_t, v_t)                  # [B,H,d] each
    outs = cache.steps(q, k, v)                      # [n,B,H,d] each
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

__all__ = ["H2OCache", "H2OError", "lib", "LIB_PATH", "HEADER_PATH", "declared_functions", "kernel_arch", "probe_read_gbs"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libh2o.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "h2o.h")

H2O_F32, H2O_BF16, H2O_BF16_FP8KV = 0, 1, 2
_STATUS = {0: "H2O_OK", 1: "H2O_EINVAL", 2: "H2O_ESTATE", 3: "H2O_ECUDA", 4: "H2O_ENOMEM",
           5: "H2O_EDEVICE", 6: "H2O_EUNSUPPORTED"}

_lib = None


class H2OError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = _STATUS.get(status, str(status))
        extra = ""
        if status == 3 and _lib is not None:
            extra = f" (cuda error {_lib.h2o_last_cuda_error()})"
        super().__init__(f"{what}: {name}{extra}")


def declared_functions():
    """Names of the functions include/h2o.h declares."""
    txt = open(HEADER_PATH).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(h2o_[a-z0-9_]+)\s*\(", txt)))


def lib():
    """Load libh2o.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with h2o_heavy_hitter_decode_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
        L.h2o_cache_workspace_bytes.argtypes = [i32] * 6
        L.h2o_cache_workspace_bytes.restype = sz
        L.h2o_cache_create.argtypes = [i32] * 6 + [vp, vp, C.POINTER(vp)]
        L.h2o_cache_destroy.argtypes = [vp]
        L.h2o_set_stream.argtypes = [vp, vp]
        L.h2o_prefill.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp]
        L.h2o_prefill_rows.argtypes = [vp, i32, i32, vp, vp, vp, i32, vp, vp, vp]
        L.h2o_decode_step.argtypes = [vp, vp, vp, vp, vp]
        L.h2o_decode_steps.argtypes = [vp, i32, vp, vp, vp, vp, vp]
        L.h2o_cache_export.argtypes = [vp, vp, vp, vp, vp, C.POINTER(i64), C.POINTER(i32)]
        L.h2o_cache_import.argtypes = [vp, vp, vp, vp, vp, i64, i32]
        L.h2o_cache_info.argtypes = [vp] + [C.POINTER(i32)] * 6 + [C.POINTER(i64)] + [C.POINTER(i32)] * 2
        L.h2o_get_error.argtypes = [vp]
        L.h2o_profile_enable.argtypes = [vp, i32]
        L.h2o_set_decode_form.argtypes = [vp, i32]
        L.h2o_decode_form_used.argtypes = [vp, C.POINTER(i32)]
        L.h2o_cache_set_policy.argtypes = [vp, i32, i32]
        L.h2o_cache_export_scales.argtypes = [vp, vp, vp]
        L.h2o_cache_import_scales.argtypes = [vp, vp, vp]
        L.h2o_cache_get_policy.argtypes = [vp, C.POINTER(i32), C.POINTER(i32)]
        L.h2o_profile_read.argtypes = [vp, C.POINTER(C.c_double), C.POINTER(i64)]
        L.h2o_status_str.argtypes = [i32]
        L.h2o_status_str.restype = C.c_char_p
        L.h2o_last_cuda_error.restype = i32
        L.h2o_build_arch.restype = i32
        L.h2o_probe_read.argtypes = [vp, sz, i32, vp, vp]
        L.h2o_probe_read.restype = i32
        L.h2o_kernel_arch.argtypes = [C.POINTER(i32), C.POINTER(i32)]
        L.h2o_kernel_arch.restype = i32
        for f in ("h2o_cache_create", "h2o_cache_destroy", "h2o_set_stream", "h2o_prefill", "h2o_prefill_rows",
                  "h2o_decode_step",
                  "h2o_decode_steps", "h2o_cache_export", "h2o_cache_import", "h2o_cache_info",
                  "h2o_get_error", "h2o_profile_enable", "h2o_profile_read", "h2o_set_decode_form",
                  "h2o_decode_form_used", "h2o_cache_set_policy", "h2o_cache_get_policy",
                  "h2o_cache_export_scales", "h2o_cache_import_scales"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def kernel_arch():
    """(ptx_version, binary_version) of the library's kernels as loaded on
    the current device (103, 103 for the sm_103a build)."""
    ptx, binv = C.c_int32(), C.c_int32()
    _check(lib().h2o_kernel_arch(C.byref(ptx), C.byref(binv)), "h2o_kernel_arch")
    return ptx.value, binv.value


def probe_read_gbs(nbytes: int, reps: int = 50, device=None) -> float:
    """Read bandwidth (GB/s) of a device buffer of `nbytes`, measured with the
    library's read kernel (h2o_probe_read): `reps` sweeps after a warm-up,
    timed with CUDA events on the current stream."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    n = max(16, int(nbytes) // 16 * 16)
    buf = torch.ones(n // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev)
    run = lambda r: _check(lib().h2o_probe_read(_ptr(buf), n, int(r), _ptr(sink), C.c_void_p(s.cuda_stream)),
                           "h2o_probe_read")
    run(2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    run(reps)
    e1.record(s)
    e1.synchronize()
    return n * reps / (e0.elapsed_time(e1) / 1e3) / 1e9


def _check(rc: int, what: str):
    if rc != 0:
        raise H2OError(rc, what)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _dt(dtype) -> int:
    if dtype == torch.bfloat16:
        return H2O_BF16
    if dtype == torch.float32:
        return H2O_F32
    raise TypeError(f"unsupported dtype {dtype}: use torch.bfloat16 or torch.float32")


class H2OCache:
    """Per-(batch, head) H2O caches of k = k_heavy + k_local slots.

    The workspace (K/V slots, position tags, scores, split partials) is one
    torch uint8 tensor owned by this object.  Calls enqueue on torch's current
    CUDA stream."""

    def __init__(self, B: int, H: int, d: int, k_heavy: int, k_local: int, dtype=torch.bfloat16,
                 device=None, kv_fp8: bool = False):
        """``dtype`` is the type of every input and output; ``kv_fp8`` (bf16
        only) stores the K/V slots as e4m3 codes with one fp32 scale per row
        (H2O_BF16_FP8KV)."""
        L = lib()
        self.B, self.H, self.d, self.k_heavy, self.k_local = B, H, d, k_heavy, k_local
        self.k = k_heavy + k_local
        self.dtype = dtype
        self.kv_fp8 = bool(kv_fp8)
        if self.kv_fp8 and dtype != torch.bfloat16:
            raise TypeError("an fp8 K/V cache takes bf16 inputs")
        code = H2O_BF16_FP8KV if self.kv_fp8 else _dt(dtype)
        self.kv_dtype = torch.float8_e4m3fn if self.kv_fp8 else dtype
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        if self.device.type != "cuda":
            raise ValueError("H2OCache lives on a CUDA device")
        with torch.cuda.device(self.device):
            nbytes = L.h2o_cache_workspace_bytes(B, H, d, k_heavy, k_local, code)
            if nbytes == 0:
                raise H2OError(1, f"h2o_cache_workspace_bytes({B},{H},{d},{k_heavy},{k_local})")
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            h = C.c_void_p()
            _check(L.h2o_cache_create(B, H, d, k_heavy, k_local, code, _ptr(self.workspace),
                                      C.c_void_p(torch.cuda.current_stream(self.device).cuda_stream),
                                      C.byref(h)), "h2o_cache_create")
            self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.h2o_cache_destroy(h)
            self._h = None

    # -------------------------------------------------------------- helpers
    def _sync_stream(self):
        _check(lib().h2o_set_stream(self._h, C.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)),
               "h2o_set_stream")

    def _arg(self, t, shape, name, dtype=None):
        dtype = self.dtype if dtype is None else dtype
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a tensor")
        if t.device != self.device or t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)} on {self.device}, got "
                             f"{t.dtype} {tuple(t.shape)} on {t.device} (contiguous={t.is_contiguous()})")
        return t

    # ---------------------------------------------------------------- calls
    def prefill(self, Q, K, V, O=None, lse=None, colsum=None, want_O=True):
        """Causal prefill over the prompt; returns (O, lse, colsum)."""
        B, H, d = self.B, self.H, self.d
        Lp = Q.shape[2]
        shp = (B, H, Lp, d)
        self._arg(Q, shp, "Q"); self._arg(K, shp, "K"); self._arg(V, shp, "V")
        if O is None and want_O:
            O = torch.empty(shp, dtype=self.dtype, device=self.device)
        if O is not None:
            self._arg(O, shp, "O")
        if lse is None:
            lse = torch.empty((B, H, Lp), dtype=torch.float32, device=self.device)
        if colsum is None:
            colsum = torch.empty((B, H, Lp), dtype=torch.float32, device=self.device)
        self._arg(lse, (B, H, Lp), "lse", torch.float32)
        self._arg(colsum, (B, H, Lp), "colsum", torch.float32)
        self._sync_stream()
        _check(lib().h2o_prefill(self._h, _ptr(Q), _ptr(K), _ptr(V), int(Lp), _ptr(O), _ptr(lse), _ptr(colsum)),
               "h2o_prefill")
        return O, lse, colsum

    def prefill_rows(self, b0: int, Q, K, V, O=None, lse=None, colsum=None, want_O=True):
        """Prefill of batch rows b0 .. b0+nb-1 (nb = Q.shape[0]); returns
        (O, lse, colsum) of those rows.  Decode may start once every row is
        prefilled, all with the same prompt length."""
        nb, H, d = Q.shape[0], self.H, self.d
        Lp = Q.shape[2]
        shp = (nb, H, Lp, d)
        self._arg(Q, shp, "Q"); self._arg(K, shp, "K"); self._arg(V, shp, "V")
        if O is None and want_O:
            O = torch.empty(shp, dtype=self.dtype, device=self.device)
        if O is not None:
            self._arg(O, shp, "O")
        if lse is None:
            lse = torch.empty((nb, H, Lp), dtype=torch.float32, device=self.device)
        if colsum is None:
            colsum = torch.empty((nb, H, Lp), dtype=torch.float32, device=self.device)
        self._arg(lse, (nb, H, Lp), "lse", torch.float32)
        self._arg(colsum, (nb, H, Lp), "colsum", torch.float32)
        self._sync_stream()
        _check(lib().h2o_prefill_rows(self._h, int(b0), int(nb), _ptr(Q), _ptr(K), _ptr(V), int(Lp), _ptr(O),
                                      _ptr(lse), _ptr(colsum)), "h2o_prefill_rows")
        return O, lse, colsum

    def step(self, q, k, v, out=None):
        shp = (self.B, self.H, self.d)
        self._arg(q, shp, "q"); self._arg(k, shp, "k"); self._arg(v, shp, "v")
        if out is None:
            out = torch.empty(shp, dtype=self.dtype, device=self.device)
        self._arg(out, shp, "out")
        self._sync_stream()
        _check(lib().h2o_decode_step(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(out)), "h2o_decode_step")
        return out

    def steps(self, q, k, v, out=None, evicted=None):
        """n decode steps; q, k, v [n,B,H,d]; returns out (and fills evicted [n,B,H] int32 if given)."""
        n = q.shape[0]
        shp = (n, self.B, self.H, self.d)
        self._arg(q, shp, "q"); self._arg(k, shp, "k"); self._arg(v, shp, "v")
        if out is None:
            out = torch.empty(shp, dtype=self.dtype, device=self.device)
        self._arg(out, shp, "out")
        if evicted is not None:
            self._arg(evicted, (n, self.B, self.H), "evicted", torch.int32)
        self._sync_stream()
        _check(lib().h2o_decode_steps(self._h, int(n), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(evicted)),
               "h2o_decode_steps")
        return out

    def export(self):
        """Copy of the cache state: dict(pos, score, K, V, next_pos, n_valid),
        plus K_scale, V_scale [B,H,k] for an fp8 cache (K, V then hold the
        e4m3 codes as torch.float8_e4m3fn)."""
        B, H, k, d = self.B, self.H, self.k, self.d
        pos = torch.empty((B, H, k), dtype=torch.int32, device=self.device)
        score = torch.empty((B, H, k), dtype=torch.float32, device=self.device)
        K = torch.empty((B, H, k, d), dtype=self.kv_dtype, device=self.device)
        V = torch.empty_like(K)
        nxt, nv = C.c_int64(), C.c_int32()
        self._sync_stream()
        _check(lib().h2o_cache_export(self._h, _ptr(pos), _ptr(score), _ptr(K), _ptr(V), C.byref(nxt), C.byref(nv)),
               "h2o_cache_export")
        out = dict(pos=pos, score=score, K=K, V=V, next_pos=nxt.value, n_valid=nv.value)
        if self.kv_fp8:
            out["K_scale"] = torch.empty((B, H, k), dtype=torch.float32, device=self.device)
            out["V_scale"] = torch.empty_like(out["K_scale"])
            _check(lib().h2o_cache_export_scales(self._h, _ptr(out["K_scale"]), _ptr(out["V_scale"])),
                   "h2o_cache_export_scales")
        return out

    def import_state(self, pos, score, K, V, next_pos: int, n_valid: int, K_scale=None, V_scale=None):
        """Replace the state (layouts of export; an fp8 cache also needs the
        row scales)."""
        B, H, k, d = self.B, self.H, self.k, self.d
        self._arg(pos, (B, H, k), "pos", torch.int32)
        self._arg(score, (B, H, k), "score", torch.float32)
        self._arg(K, (B, H, k, d), "K", self.kv_dtype); self._arg(V, (B, H, k, d), "V", self.kv_dtype)
        if self.kv_fp8:
            self._arg(K_scale, (B, H, k), "K_scale", torch.float32)
            self._arg(V_scale, (B, H, k), "V_scale", torch.float32)
        self._sync_stream()
        _check(lib().h2o_cache_import(self._h, _ptr(pos), _ptr(score), _ptr(K), _ptr(V), int(next_pos), int(n_valid)),
               "h2o_cache_import")
        if self.kv_fp8:
            _check(lib().h2o_cache_import_scales(self._h, _ptr(K_scale), _ptr(V_scale)), "h2o_cache_import_scales")

    def info(self):
        vals = [C.c_int32() for _ in range(6)]
        nxt = C.c_int64()
        nv, ns = C.c_int32(), C.c_int32()
        _check(lib().h2o_cache_info(self._h, *[C.byref(x) for x in vals], C.byref(nxt), C.byref(nv), C.byref(ns)),
               "h2o_cache_info")
        B, H, d, kh, kl, dt = (x.value for x in vals)
        return dict(B=B, H=H, d=d, k_heavy=kh, k_local=kl, dtype=dt, next_pos=nxt.value, n_valid=nv.value,
                    n_split=ns.value)

    PHASES = ("prefill_attn", "prefill_colsum", "prefill_select", "decode")
    DECODE_FORMS = {"auto": 0, "per_step": 1, "cooperative": 2, "cluster": 3, "pipelined": 4}

    def set_decode_form(self, form):
        """How multi-step decode runs: "auto", "per_step", "cooperative",
        "cluster" or "pipelined" (see h2o_set_decode_form)."""
        f = self.DECODE_FORMS[form] if isinstance(form, str) else int(form)
        _check(lib().h2o_set_decode_form(self._h, f), "h2o_set_decode_form")

    def decode_form_used(self) -> str:
        """Form of the last decode call: "per_step", "cooperative", "cluster", "pipelined" or "" (none yet)."""
        f = C.c_int32()
        _check(lib().h2o_decode_form_used(self._h, C.byref(f)), "h2o_decode_form_used")
        return {0: "", 1: "per_step", 2: "cooperative", 3: "cluster", 4: "pipelined"}[f.value]

    def set_policy(self, n_sink: int = 0, score_mode: int = 0):
        """Eviction variant for later calls: ``n_sink`` pinned first positions
        (0 <= n_sink <= k_heavy) and ``score_mode`` 1 to rank by mean weight
        instead of summed weight (see h2o_cache_set_policy)."""
        _check(lib().h2o_cache_set_policy(self._h, int(n_sink), int(score_mode)), "h2o_cache_set_policy")

    def policy(self):
        """(n_sink, score_mode) of this cache."""
        ns, sm = C.c_int32(), C.c_int32()
        _check(lib().h2o_cache_get_policy(self._h, C.byref(ns), C.byref(sm)), "h2o_cache_get_policy")
        return ns.value, sm.value

    def profile(self, on: bool = True):
        """Bracket each phase with CUDA events on the cache's stream."""
        _check(lib().h2o_profile_enable(self._h, 1 if on else 0), "h2o_profile_enable")

    def profile_read(self):
        """{phase: (milliseconds, kernel launches)} since the last read."""
        ms = (C.c_double * 4)()
        n = (C.c_int64 * 4)()
        _check(lib().h2o_profile_read(self._h, ms, n), "h2o_profile_read")
        return {p: (ms[i], n[i]) for i, p in enumerate(self.PHASES)}

    def check_device_error(self):
        self._sync_stream()
        _check(lib().h2o_get_error(self._h), "h2o_get_error")
