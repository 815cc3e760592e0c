"""Python binding of libqidit.so, the GB300 Qwen-Image-2.1 DiT step library.

Argument marshalling only: every step of the DiT pass runs in the library's
CUDA kernels. Tensors are torch tensors (device memory and streams come from
PyTorch); the calls mirror include/qidit.h one to one. There is no fallback:
if the library is missing or fails to load, `lib()` raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB, build  # noqa: F401  (build() compiles the library)

HIDDEN = 4096
HEADS = 32
HEAD_DIM = 128
FFN = 12288
PATCH = 64
TDIM = 256
ROPE_COLS = 64
NPOS = 9216
STEP_JOINT = 0
STEP_USE_CACHE = 1
STEP_HOST_IO = 2
PROF_CLASSES = ("qkv_gemm", "attention", "out_gemm", "gateup_gemm", "down_gemm", "other")
RANGE_KINDS = ("x_mod1", "q_rope", "k_rope", "v", "o", "x_mod2", "h", "txt_in")

STATUS = {
    0: "QI_OK", 1: "QI_ERR_INVALID_ARG", 2: "QI_ERR_SHAPE", 3: "QI_ERR_STATE", 4: "QI_ERR_OOM",
    5: "QI_ERR_CUDA", 6: "QI_ERR_DEVICE_TIMEOUT", 7: "QI_ERR_NOT_IMPLEMENTED", 8: "QI_ERR_NONFINITE",
}

# every symbol include/qidit.h declares
SYMBOLS = (
    "qi_dit_create", "qi_dit_destroy", "qi_dit_load_global", "qi_dit_load_block",
    "qi_rope_axis_tables", "qi_rope_tables", "qi_flow_sigmas", "qi_pack_noise", "qi_euler_update",
    "qi_dit_step", "qi_text_kv_capture", "qi_kv_cache_bytes", "qi_dit_check",
    "qi_dit_block_forward", "qi_dit_read_kv", "qi_dit_set_trace", "qi_dit_profile", "qi_dit_profile_classes",
    "qi_dit_profile_read", "qi_last_error", "qi_gemm_bf16", "qi_attention_f16", "qi_gemm_bf16_noalloc", "qi_gemv_bf16",
    "qi_dit_step_cfg", "qi_dpmpp2m_coeffs", "qi_dpmpp2m_update", "qi_dit_step_fbcache", "qi_dit_fbcache_reset",
    "qi_dit_set_mxfp8", "qi_quant_mxfp8", "qi_gemm_mxfp8", "qi_debug_inject", "qi_dit_euler_step", "qi_dit_set_range_probe",
)


class QiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class DitConfig(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_int), ("L_max", ctypes.c_int), ("N_max", ctypes.c_int), ("kv_slots", ctypes.c_int),
                ("mxfp8", ctypes.c_int)]


_GLOBAL_FIELDS = ("t_w1", "t_b1", "t_w2", "t_b2", "mod_w", "mod_b", "txt_norm_w", "txt_w", "txt_b",
                  "img_w", "img_b", "out_w", "out_b")
_BLOCK_FIELDS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


class GlobalWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _GLOBAL_FIELDS]


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _BLOCK_FIELDS]


class SchedParams(ctypes.Structure):
    _fields_ = [("base_shift", ctypes.c_double), ("max_shift", ctypes.c_double), ("base_seq", ctypes.c_int),
                ("max_seq", ctypes.c_int), ("shift_terminal", ctypes.c_double), ("train_steps", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libqidit.so (built in-tree by build()); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("QIDIT_LIB", LIB)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run diffusion_transformer_text_gb300.build() first")
    L = ctypes.CDLL(path)
    P, I, F, U, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint, ctypes.c_size_t
    sig = {
        "qi_dit_create": [ctypes.POINTER(DitConfig), I, ctypes.POINTER(P)],
        "qi_dit_destroy": [P],
        "qi_dit_load_global": [P, ctypes.POINTER(GlobalWeights), I, P],
        "qi_dit_load_block": [P, I, ctypes.POINTER(BlockWeights), I, P],
        "qi_rope_axis_tables": [F, P, P, P, P, P, P, P],
        "qi_rope_tables": [I, I, I, F, P, P, P, P, P],
        "qi_flow_sigmas": [I, I, ctypes.POINTER(SchedParams), P, P],
        "qi_pack_noise": [P, I, I, P, P],
        "qi_euler_update": [P, P, I, F, F, P],
        "qi_dit_step": [P, P, I, P, I, F, P, P, P, P, P, U, P],
        "qi_dit_euler_step": [P, P, I, P, I, F, F, F, P, P, P, P, P, U, P],
        "qi_text_kv_capture": [P, P, I, P, P, P],
        "qi_dit_check": [P, P],
        "qi_dit_block_forward": [P, I, P, I, I, F, P, P, P],
        "qi_dit_read_kv": [P, I, I, I, P, P, P],
        "qi_dit_set_trace": [P, I, I, P],
        "qi_dit_set_range_probe": [P, P],
        "qi_dit_profile": [P, I],
        "qi_dit_profile_classes": [P, U, I],
        "qi_dit_profile_read": [P, P, P],
        "qi_gemm_bf16": [P, P, P, P, I, I, I, P],
        "qi_attention_f16": [P, P, P, P, I, I, I, I, P],
        "qi_gemv_bf16": [P, I, P, P, I, P, I, P],
        "qi_gemm_bf16_noalloc": [P, P, P, I, I, I, I, P],
        "qi_dit_step_cfg": [P, P, I, F, F, P, I, P, P, P, P, P, I, P, P, P, P, P, U, P],
        "qi_dpmpp2m_coeffs": [P, I, I, P, P],
        "qi_dit_step_fbcache": [P, P, I, P, I, F, P, P, P, P, F, P, P, P, U, P],
        "qi_dit_fbcache_reset": [P],
        "qi_dit_set_mxfp8": [P, I],
        "qi_debug_inject": [P, I, I],
        "qi_quant_mxfp8": [P, I, I, I, P, P, P],
        "qi_gemm_mxfp8": [P, P, P, P, P, P, I, I, I, P],
        "qi_dpmpp2m_update": [P, P, P, I, P, I, I, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.qi_kv_cache_bytes.argtypes = [I, I]
    L.qi_kv_cache_bytes.restype = S
    L.qi_last_error.argtypes = []
    L.qi_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int):
    if status != 0:
        raise QiError(status, lib().qi_last_error().decode())


def _ptr(t) -> int | None:
    """Device pointer of a contiguous torch tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev_f32(t, shape, name):
    import torch
    if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: want float32 cuda {tuple(shape)}, got {t.dtype} {t.device} {tuple(t.shape)}")
    return _ptr(t)


# ---------------------------------------------------------------- host contract


def kv_cache_bytes(blocks: int, L: int) -> int:
    return int(lib().qi_kv_cache_bytes(blocks, L))


def flow_sigmas(steps: int, N: int, params: dict | None = None):
    """(sigmas float32 [steps+1], timesteps float32 [steps]), computed by the library on the host."""
    sig = np.zeros(steps + 1, np.float32)
    ts = np.zeros(max(steps, 1), np.float32)
    p = None
    if params is not None:
        p = ctypes.byref(SchedParams(**params))
    _check(lib().qi_flow_sigmas(steps, N, p, sig.ctypes.data, ts.ctypes.data))
    return sig, ts[:steps]


def rope_axis_tables(theta: float = 10000.0, device="cuda"):
    """[(cos0, sin0) [9216, 8], (cos1, sin1) [9216, 28], (cos2, sin2) [9216, 28]] on the device."""
    import torch
    out = [(torch.empty(NPOS, w, device=device), torch.empty(NPOS, w, device=device)) for w in (8, 28, 28)]
    _check(lib().qi_rope_axis_tables(theta, *[_ptr(t) for pair in out for t in pair], _stream()))
    return out


def rope_tables(L: int, h: int, w: int, theta: float = 10000.0, device="cuda"):
    """txt_cos, txt_sin [L, 64] and img_cos, img_sin [h*w, 64] on the device."""
    import torch
    tc = torch.empty(L, ROPE_COLS, device=device)
    ts = torch.empty(L, ROPE_COLS, device=device)
    ic = torch.empty(h * w, ROPE_COLS, device=device)
    is_ = torch.empty(h * w, ROPE_COLS, device=device)
    _check(lib().qi_rope_tables(L, h, w, theta, _ptr(tc), _ptr(ts), _ptr(ic), _ptr(is_), _stream()))
    return tc, ts, ic, is_


def pack_noise(z):
    """Channel-major latent z [64, h, w] (device) -> tokens [h*w, 64]."""
    import torch
    c, h, w = z.shape
    x = torch.empty(h * w, c, device=z.device, dtype=torch.float32)
    _dev_f32(z, (PATCH, h, w), "z")
    _check(lib().qi_pack_noise(_ptr(z), h, w, _ptr(x), _stream()))
    return x


def euler_update(x, vel, sigma_i: float, sigma_next: float):
    """In place: x <- x + (sigma_next - sigma_i) * vel (float32, no FMA)."""
    N = x.shape[0]
    _dev_f32(x, (N, PATCH), "x")
    _dev_f32(vel, (N, PATCH), "vel")
    _check(lib().qi_euler_update(_ptr(x), _ptr(vel), N, sigma_i, sigma_next, _stream()))
    return x


def _host_sigmas(sigmas):
    import numpy as np
    s = np.ascontiguousarray(np.asarray(sigmas, dtype=np.float32))
    return s, s.ctypes.data_as(ctypes.c_void_p)


def dpmpp2m_coeffs(sigmas, i: int):
    """Host-side coefficients of DPM++ 2M step i: (order, a, b, c0, c1) as float32 values."""
    import numpy as np
    s, sp = _host_sigmas(sigmas)
    order = ctypes.c_int(-1)
    c = np.zeros(4, np.float32)
    _check(lib().qi_dpmpp2m_coeffs(sp, len(s) - 1, i, ctypes.byref(order), c.ctypes.data_as(ctypes.c_void_p)))
    return (order.value, *[np.float32(v) for v in c])


def dpmpp2m_update(x, vel, d_prev, sigmas, i: int):
    """In place: DPM++ 2M step i on x [N, 64]; d_prev [N, 64] carries D between steps."""
    N = x.shape[0]
    _dev_f32(x, (N, PATCH), "x")
    _dev_f32(vel, (N, PATCH), "vel")
    _dev_f32(d_prev, (N, PATCH), "d_prev")
    s, sp = _host_sigmas(sigmas)
    _check(lib().qi_dpmpp2m_update(_ptr(x), _ptr(vel), _ptr(d_prev), N, sp, len(s) - 1, i, _stream()))
    return x


def debug_inject(kind: int, arg: int = 0, dit=None):
    """Test hook: 1 = fail the arg-th next device allocation; 2 = stall the next block GEMM
    of `dit` until its bounded wait expires; 0 = cancel."""
    _check(lib().qi_debug_inject(dit._h if dit is not None else None, kind, arg))


def quant_mxfp8(x, bf16: bool):
    """MXFP8 along the last axis of a [rows, K] 16-bit device tensor (bf16 bits or fp16):
    returns (E4M3 bytes [rows, K] uint8, scale chunks uint8)."""
    import torch
    rows, K = x.shape
    q = torch.empty(rows, K, dtype=torch.uint8, device=x.device)
    sf = torch.zeros(((rows + 127) // 128) * (K // 128) * 512, dtype=torch.uint8, device=x.device)
    _check(lib().qi_quant_mxfp8(_ptr(x), int(bf16), rows, K, _ptr(q), _ptr(sf), _stream()))
    return q, sf


def attention(q, k, v, L: int, q_off: int = 0, Lk: int | None = None):
    """Test hook: block-causal attention, fp16 q [Rq, 4096], k/v [Lk, 4096] -> o [Rq, 4096]."""
    import torch
    Rq = q.shape[0]
    Lk = k.shape[0] if Lk is None else Lk
    o = torch.empty(Rq, HIDDEN, dtype=q.dtype, device=q.device)
    _check(lib().qi_attention_f16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), Rq, q_off, L, Lk, _stream()))
    return o


def gemv(x, W, b, silu_in: bool = False):
    """Test hook: the two-row GEMV of the timestep MLP and the shared modulation.
    x fp32 [2, in_dim], W bf16 bits [out_dim, in_dim], b bf16 bits [out_dim] -> y fp32 [2, out_dim]."""
    import torch
    out_dim, in_dim = W.shape
    y = torch.empty(2, out_dim, dtype=torch.float32, device=x.device)
    _check(lib().qi_gemv_bf16(_ptr(x), in_dim, _ptr(W), _ptr(b), out_dim, _ptr(y), int(silu_in), _stream()))
    return y


# ---------------------------------------------------------------- the DiT


class DiT:
    """A qi_dit handle: bf16 weight store, activations and per-block text K/V."""

    def __init__(self, blocks: int = 32, L_max: int = 512, N_max: int = 4096, device: int = 0, kv_slots: int = 1,
                 mxfp8: bool = False):
        self.blocks, self.L_max, self.N_max, self.device = blocks, L_max, N_max, device
        h = ctypes.c_void_p()
        cfg = DitConfig(blocks, L_max, N_max, kv_slots, int(mxfp8))
        _check(lib().qi_dit_create(ctypes.byref(cfg), device, ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().qi_dit_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _src(arr):
        """(pointer, on_device, keepalive) for a numpy uint16 or torch tensor."""
        if isinstance(arr, np.ndarray):
            a = np.ascontiguousarray(arr)
            if a.dtype != np.uint16:
                raise ValueError("weights must be bf16 bit patterns (uint16)")
            return a.ctypes.data, 0, a
        t = arr.contiguous()
        return t.data_ptr(), int(t.is_cuda), t

    def load_global(self, g: dict):
        srcs = [self._src(g[n]) for n in _GLOBAL_FIELDS]
        on_dev = {s[1] for s in srcs}
        if len(on_dev) != 1:
            raise ValueError("mixed host/device weight sources")
        gw = GlobalWeights(*[s[0] for s in srcs])
        _check(lib().qi_dit_load_global(self._h, ctypes.byref(gw), on_dev.pop(), _stream()))

    def load_block(self, b: int, w: dict):
        srcs = [self._src(w[n]) for n in _BLOCK_FIELDS]
        on_dev = {s[1] for s in srcs}
        if len(on_dev) != 1:
            raise ValueError("mixed host/device weight sources")
        bw = BlockWeights(*[s[0] for s in srcs])
        _check(lib().qi_dit_load_block(self._h, b, ctypes.byref(bw), on_dev.pop(), _stream()))

    def step(self, img_tokens, txt_feats, timestep: float, txt_cos, txt_sin, img_cos, img_sin,
             use_cache: bool = False, vel=None, stream=None):
        """One DiT pass on device tensors; returns vel [N, 64] (float32, device)."""
        import torch
        N = img_tokens.shape[0]
        L = txt_cos.shape[0] if txt_cos is not None else txt_feats.shape[0]
        _dev_f32(img_tokens, (N, PATCH), "img_tokens")
        _dev_f32(img_cos, (N, ROPE_COLS), "img_cos")
        _dev_f32(img_sin, (N, ROPE_COLS), "img_sin")
        if not use_cache:
            _dev_f32(txt_feats, (L, HIDDEN), "txt_feats")
            _dev_f32(txt_cos, (L, ROPE_COLS), "txt_cos")
            _dev_f32(txt_sin, (L, ROPE_COLS), "txt_sin")
        if vel is None:
            vel = torch.empty(N, PATCH, device=img_tokens.device, dtype=torch.float32)
        flags = STEP_USE_CACHE if use_cache else STEP_JOINT
        _check(lib().qi_dit_step(self._h, _ptr(img_tokens), N, _ptr(txt_feats) if not use_cache else None, L,
                                 float(timestep), _ptr(txt_cos) if not use_cache else None,
                                 _ptr(txt_sin) if not use_cache else None, _ptr(img_cos), _ptr(img_sin),
                                 _ptr(vel), flags, _stream(stream)))
        return vel

    def step_cached(self, img_tokens, L: int, timestep: float, img_cos, img_sin, vel=None, stream=None):
        """Image-only pass over the stored text K/V of a prompt of length L."""
        import torch
        N = img_tokens.shape[0]
        _dev_f32(img_tokens, (N, PATCH), "img_tokens")
        if vel is None:
            vel = torch.empty(N, PATCH, device=img_tokens.device, dtype=torch.float32)
        _check(lib().qi_dit_step(self._h, _ptr(img_tokens), N, None, L, float(timestep), None, None,
                                 _ptr(img_cos), _ptr(img_sin), _ptr(vel), STEP_USE_CACHE, _stream(stream)))
        return vel

    def step_host(self, img_tokens, txt_feats, L: int, timestep: float, txt_cos, txt_sin, img_cos, img_sin,
                  vel, use_cache: bool = False, stream=None):
        """Same pass with HOST buffers (numpy or pinned torch CPU tensors); copies happen in the call."""
        def hp(a):
            if a is None:
                return None
            if isinstance(a, np.ndarray):
                return a.ctypes.data
            return a.data_ptr()
        N = img_tokens.shape[0]
        flags = STEP_HOST_IO | (STEP_USE_CACHE if use_cache else 0)
        _check(lib().qi_dit_step(self._h, hp(img_tokens), N, hp(txt_feats), L, float(timestep), hp(txt_cos),
                                 hp(txt_sin), hp(img_cos), hp(img_sin), hp(vel), flags, _stream(stream)))
        return vel

    def euler_step(self, x, txt_feats, L: int, timestep: float, sigma_i: float, sigma_next: float, txt_cos, txt_sin,
                   img_cos, img_sin, use_cache: bool = False, vel=None, stream=None):
        """One sampler step on device tensors: the DiT pass on x [N, 64], then x += (sigma_next - sigma_i) * vel
        in place. txt_* may be None with use_cache. vel (optional, [N, 64]) receives the velocity."""
        N = x.shape[0]
        _dev_f32(x, (N, PATCH), "x")
        _dev_f32(img_cos, (N, ROPE_COLS), "img_cos")
        _dev_f32(img_sin, (N, ROPE_COLS), "img_sin")
        if not use_cache:
            _dev_f32(txt_feats, (L, HIDDEN), "txt_feats")
            _dev_f32(txt_cos, (L, ROPE_COLS), "txt_cos")
            _dev_f32(txt_sin, (L, ROPE_COLS), "txt_sin")
        if vel is not None:
            _dev_f32(vel, (N, PATCH), "vel")
        flags = STEP_USE_CACHE if use_cache else STEP_JOINT
        _check(lib().qi_dit_euler_step(self._h, _ptr(x), N, None if use_cache else _ptr(txt_feats), L,
                                       float(timestep), float(sigma_i), float(sigma_next),
                                       None if use_cache else _ptr(txt_cos), None if use_cache else _ptr(txt_sin),
                                       _ptr(img_cos), _ptr(img_sin), _ptr(vel), flags, _stream(stream)))
        return x

    def euler_step_host(self, x, txt_feats, L: int, timestep: float, sigma_i: float, sigma_next: float, txt_cos,
                        txt_sin, img_cos, img_sin, use_cache: bool = False, vel=None, stream=None):
        """The same sampler step on HOST buffers (numpy arrays or pinned torch CPU tensors, float32,
        contiguous): the call copies in, runs, copies x (and vel) back and synchronises."""
        def hp(a, name, shape):
            if a is None:
                return None
            if isinstance(a, np.ndarray):
                ok = a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.shape == shape
                ptr = a.ctypes.data
            else:
                import torch
                ok = a.dtype == torch.float32 and not a.is_cuda and a.is_contiguous() and tuple(a.shape) == shape
                ptr = a.data_ptr()
            if not ok:
                raise ValueError(f"{name}: want a contiguous float32 host array {shape}")
            return ptr
        N = x.shape[0]
        flags = STEP_HOST_IO | (STEP_USE_CACHE if use_cache else 0)
        t = (lambda a, n, sh: None) if use_cache else hp
        _check(lib().qi_dit_euler_step(self._h, hp(x, "x", (N, PATCH)), N, t(txt_feats, "txt_feats", (L, HIDDEN)), L,
                                       float(timestep), float(sigma_i), float(sigma_next),
                                       t(txt_cos, "txt_cos", (L, ROPE_COLS)), t(txt_sin, "txt_sin", (L, ROPE_COLS)),
                                       hp(img_cos, "img_cos", (N, ROPE_COLS)), hp(img_sin, "img_sin", (N, ROPE_COLS)),
                                       hp(vel, "vel", (N, PATCH)), flags, _stream(stream)))
        return x

    def step_cfg(self, img_tokens, timestep: float, guidance: float, pos, neg, use_cache: bool = False, vel=None,
                 stream=None):
        """Classifier-free guidance step. pos / neg: dicts with keys feats (or None
        with use_cache), L, txt_cos, txt_sin, img_cos, img_sin (device tensors)."""
        import torch
        N = img_tokens.shape[0]
        _dev_f32(img_tokens, (N, PATCH), "img_tokens")
        if vel is None:
            vel = torch.empty(N, PATCH, device=img_tokens.device, dtype=torch.float32)
        g = lambda d, k: None if use_cache and k in ("feats", "txt_cos", "txt_sin") else _ptr(d.get(k))
        _check(lib().qi_dit_step_cfg(
            self._h, _ptr(img_tokens), N, float(timestep), float(guidance),
            g(pos, "feats"), int(pos["L"]), g(pos, "txt_cos"), g(pos, "txt_sin"), _ptr(pos["img_cos"]),
            _ptr(pos["img_sin"]), g(neg, "feats"), int(neg["L"]), g(neg, "txt_cos"), g(neg, "txt_sin"),
            _ptr(neg["img_cos"]), _ptr(neg["img_sin"]), _ptr(vel), STEP_USE_CACHE if use_cache else STEP_JOINT,
            _stream(stream)))
        return vel

    def step_fbcache(self, img_tokens, txt_feats, L: int, timestep: float, txt_cos, txt_sin, img_cos, img_sin,
                     threshold: float, use_cache: bool = False, vel=None, stream=None):
        """One step under the first-block cache (txt_* may be None with use_cache).
        Returns (vel, rel_change, skipped)."""
        import torch
        N = img_tokens.shape[0]
        _dev_f32(img_tokens, (N, PATCH), "img_tokens")
        _dev_f32(img_cos, (N, ROPE_COLS), "img_cos")
        _dev_f32(img_sin, (N, ROPE_COLS), "img_sin")
        if not use_cache:
            _dev_f32(txt_feats, (L, HIDDEN), "txt_feats")
            _dev_f32(txt_cos, (L, ROPE_COLS), "txt_cos")
            _dev_f32(txt_sin, (L, ROPE_COLS), "txt_sin")
        if vel is None:
            vel = torch.empty(N, PATCH, device=img_tokens.device, dtype=torch.float32)
        rel = ctypes.c_float(0.0)
        skipped = ctypes.c_int(-1)
        _check(lib().qi_dit_step_fbcache(
            self._h, _ptr(img_tokens), N, None if use_cache else _ptr(txt_feats), L, float(timestep),
            None if use_cache else _ptr(txt_cos), None if use_cache else _ptr(txt_sin), _ptr(img_cos),
            _ptr(img_sin), float(threshold), _ptr(vel), ctypes.byref(rel), ctypes.byref(skipped),
            STEP_USE_CACHE if use_cache else STEP_JOINT, _stream(stream)))
        return vel, rel.value, bool(skipped.value)

    def fbcache_reset(self):
        _check(lib().qi_dit_fbcache_reset(self._h))

    def text_kv_capture(self, txt_feats, txt_cos, txt_sin, stream=None):
        L = txt_feats.shape[0]
        _dev_f32(txt_feats, (L, HIDDEN), "txt_feats")
        _check(lib().qi_text_kv_capture(self._h, _ptr(txt_feats), L, _ptr(txt_cos), _ptr(txt_sin),
                                        _stream(stream)))

    def block_forward(self, b: int, hidden, L: int, t_img: float, cos, sin, stream=None):
        """One block, joint layout, in place on hidden [L + N, 4096] (float32, device)."""
        R = hidden.shape[0]
        _dev_f32(hidden, (R, HIDDEN), "hidden")
        _dev_f32(cos, (R, ROPE_COLS), "cos")
        _dev_f32(sin, (R, ROPE_COLS), "sin")
        _check(lib().qi_dit_block_forward(self._h, b, _ptr(hidden), L, R - L, float(t_img), _ptr(cos), _ptr(sin),
                                          _stream(stream)))
        return hidden

    def read_kv(self, b: int, row0: int, rows: int):
        """(K, V) int16-viewed fp16 bits [rows, 4096] of block b (device copies)."""
        import torch
        k = torch.empty(rows, HIDDEN, dtype=torch.int16, device=f"cuda:{self.device}")
        v = torch.empty_like(k)
        _check(lib().qi_dit_read_kv(self._h, b, row0, rows, _ptr(k), _ptr(v), _stream()))
        return k, v

    def gemm(self, A, B):
        """Test hook: D = A @ B^T on the tensor-core GEMM; A [M,K], B [N,K] bf16 (int16 bits ok)."""
        import torch
        M, K = A.shape
        N = B.shape[0]
        D = torch.empty(M, N, dtype=torch.float32, device=A.device)
        _check(lib().qi_gemm_bf16(self._h, _ptr(A), _ptr(B), _ptr(D), M, N, K, _stream()))
        return D

    def gemm_mxfp8(self, A, A_sf, B, B_sf, M: int, N: int, K: int):
        """Test hook: the block-scaled GEMM on operands from quant_mxfp8; D [M, N] float32."""
        import torch
        D = torch.empty(M, N, dtype=torch.float32, device=A.device)
        _check(lib().qi_gemm_mxfp8(self._h, _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), _ptr(D), M, N, K, _stream()))
        return D

    def set_mxfp8(self, on: bool):
        """Run later passes on MXFP8 block GEMMs (handle created with mxfp8=True)."""
        _check(lib().qi_dit_set_mxfp8(self._h, int(on)))

    def set_range_probe(self, out=None):
        """Test hook: while `out` (float32 cuda [blocks, 8], zeroed) is set, passes fold the largest
        |value| of each fp16 operand per block into it (kinds in RANGE_KINDS); None turns it off."""
        if out is not None:
            _dev_f32(out, (self.blocks, len(RANGE_KINDS)), "out")
        _check(lib().qi_dit_set_range_probe(self._h, _ptr(out)))

    def set_trace(self, slot: int, block: int, dst=None):
        _check(lib().qi_dit_set_trace(self._h, slot, block, _ptr(dst)))

    def check(self, stream=None):
        _check(lib().qi_dit_check(self._h, _stream(stream)))

    def profile(self, enable: bool, classes=None, block_stride: int = 1):
        """Time kernel classes with CUDA events: all of them (classes None), or only
        the named ones (names from PROF_CLASSES), the per-block ones only in blocks
        b % block_stride == 0; enable False turns timing off."""
        if not enable:
            _check(lib().qi_dit_profile(self._h, 0))
        elif classes is None and block_stride == 1:
            _check(lib().qi_dit_profile(self._h, 1))
        else:
            mask = 0
            for c in (PROF_CLASSES if classes is None else classes):
                mask |= 1 << PROF_CLASSES.index(c)
            _check(lib().qi_dit_profile_classes(self._h, mask, int(block_stride)))

    def profile_read(self) -> dict:
        ms = (ctypes.c_double * len(PROF_CLASSES))()
        n = (ctypes.c_longlong * len(PROF_CLASSES))()
        _check(lib().qi_dit_profile_read(self._h, ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(n, ctypes.c_void_p)))
        return {c: (ms[i], n[i]) for i, c in enumerate(PROF_CLASSES)}
