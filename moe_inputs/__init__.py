"""Seeded synthetic inputs for the Mixtral sparse mixture-of-experts layer.

This module is shared by the fp64 oracle (``oracle/``) and the CUDA path and
therefore holds none of the layer's arithmetic: no router, no top-K, no
softmax, no expert feed-forward and no combine.  It only produces bf16 bit
patterns (``numpy.uint16``) for the layer's inputs and weights:

* every tensor is a counter-based stream: element ``c`` of the stream keyed by
  ``(seed, tensor, a, b)`` is ``table[mix32(...) >> 16]`` (see ``gen.c``);
* ``table`` holds the 65536 bf16-rounded quantiles ``scale * Phi^-1((u+.5)/2^16)``
  of a centred normal, so every stream is N(0, scale^2) quantised to 2^16
  equiprobable levels (tails cut at about 4.3 sigma);
* Mixtral shapes come from Table 1 of "Mixtral of Experts" (dim 4096,
  hidden_dim 14336, num_experts 8, top_k_experts 2, n_layers 32).

Distributions: x ~ N(0, 1); W_g, W1, W3 ~ N(0, 1/dim); W2 ~ N(0, 1/hidden).
Layouts (row-major): x [T, dim], W_g [dim, n], W1 and W3 [n, hidden, dim],
W2 [n, dim, hidden].

The skewed-routing workload shifts every token by one common vector ``u`` with
``u . W_g = b`` (minimum-norm solution), where the bias ``b`` is calibrated so
that, for logits distributed N(b, I), the probability that expert e is the
largest logit follows Zipf(s) over the experts.  The calibration uses the
normal distribution only, never the generated tokens.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libmoegen.so")

T_X, T_WG, T_W1, T_W3, T_W2 = 1, 2, 3, 4, 5

_lib = None
_lib_lock = threading.Lock()


def build_generator(force: bool = False) -> str:
    """Compile gen.c into libmoegen.so (gcc, OpenMP) and return its path."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            try:
                path = build_generator()
                lib = ctypes.CDLL(path)
            except (OSError, subprocess.CalledProcessError, FileNotFoundError):
                _lib = False
                return None
            lib.moegen_key.restype = ctypes.c_uint32
            lib.moegen_key.argtypes = [ctypes.c_uint32] * 4
            lib.moegen_fill.restype = None
            lib.moegen_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint32, ctypes.c_void_p]
            lib.moegen_fill_rows.restype = None
            lib.moegen_fill_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p]
            _lib = lib
        return _lib or None


# ---------------------------------------------------------------- hashing ---

def _mix32_np(x: np.ndarray) -> np.ndarray:
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(0x7FEB352D)
    x = x ^ (x >> np.uint32(15))
    x = x * np.uint32(0x846CA68B)
    x = x ^ (x >> np.uint32(16))
    return x


def stream_key(seed: int, tensor: int, a: int = 0, b: int = 0) -> int:
    """Key of the stream (seed, tensor, a, b); identical to moegen_key in gen.c."""
    with np.errstate(over="ignore"):
        k = _mix32_np(np.uint32(seed & 0xFFFFFFFF) ^ np.uint32(0x9E3779B9))
        k = _mix32_np(k ^ np.uint32(tensor))
        k = _mix32_np(k ^ np.uint32(a))
        k = _mix32_np(k ^ np.uint32(b))
    return int(k)


def _fill_np(count: int, start: int, key: int, table: np.ndarray) -> np.ndarray:
    c = np.arange(start, start + count, dtype=np.uint64)
    lo = (c & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    hi = (c >> np.uint64(32)).astype(np.uint32)
    with np.errstate(over="ignore"):
        h = _mix32_np(_mix32_np(lo ^ np.uint32(key)) ^ (hi + np.uint32(0x632BE5AB)))
    return table[h >> np.uint32(16)]


def fill(count: int, start: int, key: int, table: np.ndarray, use_c: bool = True) -> np.ndarray:
    """``count`` consecutive elements of stream ``key`` starting at counter ``start``."""
    lib = _load() if use_c else None
    if lib is None:
        return _fill_np(count, start, key, table)
    out = np.empty(count, dtype=np.uint16)
    tab = np.ascontiguousarray(table, dtype=np.uint16)
    lib.moegen_fill(out.ctypes.data, count, start, key, tab.ctypes.data)
    return out


def fill_rows(rows: np.ndarray, cols: int, key: int, table: np.ndarray) -> np.ndarray:
    """Rows ``rows`` of the [*, cols] matrix held by stream ``key``."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    lib = _load()
    if lib is None:
        out = np.empty((len(rows), cols), dtype=np.uint16)
        for i, r in enumerate(rows):
            out[i] = _fill_np(cols, int(r) * cols, key, table)
        return out
    out = np.empty((len(rows), cols), dtype=np.uint16)
    tab = np.ascontiguousarray(table, dtype=np.uint16)
    lib.moegen_fill_rows(out.ctypes.data, rows.ctypes.data, len(rows), cols, key, tab.ctypes.data)
    return out


# ------------------------------------------------------------ bf16 values ---

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(values: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


_tables: dict = {}


def normal_table(scale: float) -> np.ndarray:
    """bf16 quantile table of N(0, scale^2) over 65536 equiprobable cells."""
    key = float(scale)
    tab = _tables.get(key)
    if tab is None:
        from scipy.special import ndtri
        q = ndtri((np.arange(65536, dtype=np.float64) + 0.5) / 65536.0) * key
        tab = f32_to_bf16(q.astype(np.float32))
        _tables[key] = tab
    return tab


# ---------------------------------------------------------------- configs ---

@dataclasses.dataclass(frozen=True)
class Config:
    """One synthetic workload: shapes, seed and routing-shaping options."""
    name: str
    T: int
    dim: int
    hidden: int
    n_experts: int = 8
    top_k: int = 2
    seed: int = 46000
    layers: int = 1
    zipf_s: float = 0.0         # > 0: skew top-1 shares to Zipf(zipf_s)
    rmsnorm_eps: float = 0.0    # > 0: x <- x + MoE(RMSNorm(x)) stack

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# Table 1 of "Mixtral of Experts": dim 4096, hidden_dim 14336, 8 experts, top-2, 32 layers.
CONFIGS = {
    "tiny": Config("tiny", T=64, dim=128, hidden=256, seed=46001),
    "decode": Config("decode", T=16, dim=4096, hidden=14336, seed=46002),
    "prefill": Config("prefill", T=4096, dim=4096, hidden=14336, seed=46003),
    "skew": Config("skew", T=16384, dim=4096, hidden=14336, seed=46004, zipf_s=1.2),
    # fine-grained MoE (top 8 of 160 experts); the expert size is a reading:
    # 1/8 of a Mixtral expert, so the 8 selected experts cost one Mixtral expert
    "fine": Config("fine", T=4096, dim=4096, hidden=1792, n_experts=160, top_k=8, seed=46006),
    "fine_decode": Config("fine_decode", T=16, dim=4096, hidden=1792, n_experts=160, top_k=8,
                          seed=46007),
    "stack": Config("stack", T=8192, dim=4096, hidden=14336, seed=46005, layers=32,
                    rmsnorm_eps=1e-5),
}


def x_scale(cfg: Config) -> float:
    return 1.0


def wg_scale(cfg: Config) -> float:
    return 1.0 / np.sqrt(cfg.dim)


def w13_scale(cfg: Config) -> float:
    return 1.0 / np.sqrt(cfg.dim)


def w2_scale(cfg: Config) -> float:
    return 1.0 / np.sqrt(cfg.hidden)


def gen_router_weight(cfg: Config, layer: int = 0) -> np.ndarray:
    """W_g as bf16 bits [dim, n]."""
    key = stream_key(cfg.seed, T_WG, layer, 0)
    return fill(cfg.dim * cfg.n_experts, 0, key, normal_table(wg_scale(cfg))).reshape(
        cfg.dim, cfg.n_experts)


def gen_expert(cfg: Config, tensor: int, expert: int, layer: int = 0,
               rows: np.ndarray | None = None) -> np.ndarray:
    """One expert matrix as bf16 bits: W1/W3 [hidden, dim], W2 [dim, hidden].

    ``rows`` selects a subset of matrix rows (each row is its own counter range).
    """
    if tensor in (T_W1, T_W3):
        nr, nc, scale = cfg.hidden, cfg.dim, w13_scale(cfg)
    elif tensor == T_W2:
        nr, nc, scale = cfg.dim, cfg.hidden, w2_scale(cfg)
    else:
        raise ValueError("not an expert tensor: %r" % tensor)
    key = stream_key(cfg.seed, tensor, layer, expert)
    table = normal_table(scale)
    if rows is not None:
        return fill_rows(np.asarray(rows), nc, key, table)
    return fill(nr * nc, 0, key, table).reshape(nr, nc)


def gen_experts(cfg: Config, layer: int = 0):
    """(W1, W3, W2) as bf16 bits: [n, hidden, dim], [n, hidden, dim], [n, dim, hidden]."""
    n, d, h = cfg.n_experts, cfg.dim, cfg.hidden
    w1 = np.empty((n, h, d), np.uint16)
    w3 = np.empty((n, h, d), np.uint16)
    w2 = np.empty((n, d, h), np.uint16)
    for e in range(n):
        w1[e] = gen_expert(cfg, T_W1, e, layer)
        w3[e] = gen_expert(cfg, T_W3, e, layer)
        w2[e] = gen_expert(cfg, T_W2, e, layer)
    return w1, w3, w2


# ----------------------------------------------------------- skew shaping ---

def zipf_shares(n: int, s: float) -> np.ndarray:
    """Zipf(s) probabilities over ranks 1..n."""
    p = 1.0 / np.arange(1, n + 1, dtype=np.float64) ** s
    return p / p.sum()


def gaussian_argmax_probs(b: np.ndarray, grid: int = 4001) -> np.ndarray:
    """P(argmax_e Z_e = e) for independent Z_e ~ N(b_e, 1), by quadrature."""
    from scipy.special import ndtr
    t = np.linspace(b.min() - 9.0, b.max() + 9.0, grid)
    dt = t[1] - t[0]
    cdf = ndtr(t[None, :] - b[:, None])                     # [n, grid]
    pdf = np.exp(-0.5 * (t[None, :] - b[:, None]) ** 2) / np.sqrt(2 * np.pi)
    logc = np.log(np.maximum(cdf, 1e-300))
    others = np.exp(logc.sum(0)[None, :] - logc)            # prod over f != e
    return (pdf * others).sum(1) * dt


def calibrate_bias(shares: np.ndarray, iters: int = 200) -> np.ndarray:
    """Bias b with gaussian_argmax_probs(b) == shares (fixed-point in log space)."""
    b = np.zeros(len(shares))
    for _ in range(iters):
        p = gaussian_argmax_probs(b)
        b = b + (np.log(shares) - np.log(p))
        b -= b.mean()
    return b


def skew_shift(cfg: Config, wg_bits: np.ndarray) -> np.ndarray:
    """Common token shift u [dim] (float64) with u . W_g = b for the Zipf bias b."""
    b = calibrate_bias(zipf_shares(cfg.n_experts, cfg.zipf_s))
    wg = bf16_to_f32(wg_bits).astype(np.float64)            # [d, n]
    gram = wg.T @ wg                                        # [n, n]
    return wg @ np.linalg.solve(gram, b)                    # [d]


# ------------------------------------------------------------ activations ---

def gen_x(cfg: Config, attempt: int = 0, shift: np.ndarray | None = None) -> np.ndarray:
    """Token activations x as bf16 bits [T, dim] (stream attempt ``attempt``)."""
    key = stream_key(cfg.seed, T_X, attempt, 0)
    x = fill(cfg.T * cfg.dim, 0, key, normal_table(x_scale(cfg))).reshape(cfg.T, cfg.dim)
    if shift is not None:
        x = _apply_shift(x, shift)
    return x


def gen_x_rows(cfg: Config, rows: np.ndarray, attempt: int,
               shift: np.ndarray | None = None) -> np.ndarray:
    """Rows ``rows`` of x drawn from stream attempt ``attempt`` (used for redraws)."""
    key = stream_key(cfg.seed, T_X, attempt, 0)
    x = fill_rows(np.asarray(rows), cfg.dim, key, normal_table(x_scale(cfg)))
    if shift is not None:
        x = _apply_shift(x, shift)
    return x


def _apply_shift(x_bits: np.ndarray, shift: np.ndarray) -> np.ndarray:
    v = bf16_to_f32(x_bits).astype(np.float64) + shift[None, :]
    return f32_to_bf16(v.astype(np.float32))


@dataclasses.dataclass
class LayerInputs:
    """bf16 bit arrays of one layer: x [T,d], wg [d,n], w1/w3 [n,h,d], w2 [n,d,h]."""
    cfg: Config
    x: np.ndarray
    wg: np.ndarray
    w1: np.ndarray
    w3: np.ndarray
    w2: np.ndarray
    shift: np.ndarray | None = None


def make_layer(cfg: Config, layer: int = 0, experts: bool = True) -> LayerInputs:
    """All inputs of layer ``layer`` of workload ``cfg`` (weights optional)."""
    wg = gen_router_weight(cfg, layer)
    shift = skew_shift(cfg, wg) if cfg.zipf_s > 0 else None
    x = gen_x(cfg, 0, shift)
    if experts:
        w1, w3, w2 = gen_experts(cfg, layer)
    else:
        w1 = w3 = w2 = None
    return LayerInputs(cfg, x, wg, w1, w3, w2, shift)
