"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

Every random array comes from the Philox4x32-10 generator in ``philox.c``
(keyed by the seed, one counter stream per named tensor), so both sides of a
parity test see byte-identical inputs.  The module holds no arithmetic of the
speculative-decoding method: only draws, bf16 rounding and the shape/recipe
tables of the workloads.

Workload shapes follow the multi-token-prediction head of Qwen3.5-family
models (the head's module shape and weight inventory are listed on the
"support the qwen3_5_mtp drafter" issue page, sections "Where the MTP weights
actually live" and "Upstream contract to port").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import zlib
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile philox.c into libsynth.so (portable C, OpenMP)."""
    src = os.path.join(_HERE, "philox.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_PLANT_SO = os.path.join(_HERE, "libsynth_plant.so")
_plant = None


def build_device(force: bool = False) -> str:
    """Compile plant.cu (the benchmark's device-side target planting) for sm_103a."""
    src = os.path.join(_HERE, "plant.cu")
    if force or not os.path.exists(_PLANT_SO) or os.path.getmtime(_PLANT_SO) < os.path.getmtime(src):
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        tmp = _PLANT_SO + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc if os.path.exists(nvcc) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-O2", "-Xcompiler", "-fPIC", "-shared", src, "-o", tmp])
        os.replace(tmp, _PLANT_SO)
    return _PLANT_SO


def plant_device(stream: int, lg, vocab: int, draft, depth: int, coins, top1, top2, arg1) -> None:
    """plant_logits() on the device, in place, for one verify block (device
    pointers: lg f32 [depth+1][vocab], draft i32, coins u8, top1/top2 f32,
    arg1 i64, each [depth])."""
    global _plant
    if _plant is None:
        lib = ctypes.CDLL(build_device())
        vp = ctypes.c_void_p
        lib.synth_plant.argtypes = [vp, vp, ctypes.c_longlong, vp, ctypes.c_int, vp, vp, vp, vp]
        lib.synth_plant.restype = ctypes.c_int
        _plant = lib
    rc = _plant.synth_plant(stream, lg, vocab, draft, depth, coins, top1, top2, arg1)
    if rc != 0:
        raise RuntimeError(f"synth_plant: CUDA error {rc}")


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, u32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
        lib.synth_philox4x32_10.argtypes = [vp, vp, vp]
        lib.synth_u32.argtypes = [u64, u32, u64, vp]
        lib.synth_uniform.argtypes = [u64, u32, u64, vp]
        lib.synth_randint.argtypes = [u64, u32, u64, u32, vp]
        lib.synth_normal_f32.argtypes = [u64, u32, u64, ctypes.c_double, ctypes.c_double, vp]
        lib.synth_normal_bf16.argtypes = [u64, u32, u64, ctypes.c_double, ctypes.c_double, vp]
        lib.synth_f32_to_bf16.argtypes = [vp, u64, vp]
        _lib = lib
    return _lib


def stream_id(name: str) -> int:
    """Counter stream of a named tensor (CRC-32 of the name)."""
    return zlib.crc32(name.encode()) & 0xFFFFFFFF


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().synth_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def u32(seed: int, name: str, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    _load().synth_u32(seed, stream_id(name), n, out.ctypes.data)
    return out


def uniform(seed: int, name: str, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _load().synth_uniform(seed, stream_id(name), n, out.ctypes.data)
    return out.reshape(shape)


def randint(seed: int, name: str, shape, bound: int) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int32)
    _load().synth_randint(seed, stream_id(name), n, bound, out.ctypes.data)
    return out.reshape(shape)


def normal(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0,
           dtype: str = "f32") -> np.ndarray:
    """N(mean, std^2) draws; dtype 'f32' -> float32, 'bf16' -> uint16 bf16 bit patterns."""
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        _load().synth_normal_bf16(seed, stream_id(name), n, mean, std, out.ctypes.data)
    else:
        out = np.empty(n, dtype=np.float32)
        _load().synth_normal_f32(seed, stream_id(name), n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().synth_f32_to_bf16(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Shape:
    name: str
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    inter: int
    vocab: int
    eps: float = 1e-6
    rope_theta: float = 1e6
    dtype: str = "bf16"          # weights, KV cache and target hiddens


# Tiny fp32 head: H=256, 4 q / 2 kv heads of 64, SwiGLU 768, vocab 2048.
TINY = Shape("tiny-fp32-H256", 256, 4, 2, 64, 768, 2048, dtype="f32")
# 27B-shaped Qwen3.5-family head: H=5120, 24 q / 4 kv heads of 256, SwiGLU 17408, vocab 152064.
QWEN27B = Shape("qwen27b-shape-bf16", 5120, 24, 4, 256, 17408, 152064, dtype="bf16")


def small_shape(dtype="bf16", vocab=4096) -> Shape:
    """A reduced head of the same family, for fast multi-tile parity tests."""
    return Shape(f"small-{dtype}", 512, 8, 2, 128, 1536, vocab, dtype=dtype)


# The fifteen tensor names of the published head (raw-HF layout carries the
# "mtp." prefix; the split-out drafter layout does not).
INVENTORY = (
    "fc.weight",
    "norm.weight",
    "pre_fc_norm_embedding.weight",
    "pre_fc_norm_hidden.weight",
    "layers.0.input_layernorm.weight",
    "layers.0.post_attention_layernorm.weight",
    "layers.0.mlp.gate_proj.weight",
    "layers.0.mlp.up_proj.weight",
    "layers.0.mlp.down_proj.weight",
    "layers.0.self_attn.q_proj.weight",
    "layers.0.self_attn.k_proj.weight",
    "layers.0.self_attn.v_proj.weight",
    "layers.0.self_attn.o_proj.weight",
    "layers.0.self_attn.q_norm.weight",
    "layers.0.self_attn.k_norm.weight",
)


def tensor_shapes(s: Shape) -> dict:
    H, qw, kw, I = s.hidden, s.n_q * s.head_dim, s.n_kv * s.head_dim, s.inter
    return {
        "fc.weight": (H, 2 * H),
        "norm.weight": (H,),
        "pre_fc_norm_embedding.weight": (H,),
        "pre_fc_norm_hidden.weight": (H,),
        "layers.0.input_layernorm.weight": (H,),
        "layers.0.post_attention_layernorm.weight": (H,),
        "layers.0.mlp.gate_proj.weight": (I, H),
        "layers.0.mlp.up_proj.weight": (I, H),
        "layers.0.mlp.down_proj.weight": (H, I),
        "layers.0.self_attn.q_proj.weight": (qw, H),
        "layers.0.self_attn.k_proj.weight": (kw, H),
        "layers.0.self_attn.v_proj.weight": (kw, H),
        "layers.0.self_attn.o_proj.weight": (H, qw),
        "layers.0.self_attn.q_norm.weight": (s.head_dim,),
        "layers.0.self_attn.k_norm.weight": (s.head_dim,),
    }


@dataclass
class Model:
    shape: Shape
    tensors: dict            # name (with "mtp." prefix when raw_hf) -> np array (f32 or uint16 bf16)
    embed: np.ndarray        # [V, H], tied lm_head
    raw_hf: bool = True
    extra: dict = field(default_factory=dict)


def make_model(s: Shape, seed: int, raw_hf: bool = True, weight_std: float = 0.02,
               norm_std: float = 0.1) -> Model:
    """Weights N(0, weight_std^2); norm weights stored raw-HF as N(0, norm_std^2)
    (the +1.0 shift belongs to the loader).  With raw_hf=False the norms are
    stored pre-shifted (1 + N(0, norm_std^2)) under unprefixed names."""
    shapes = tensor_shapes(s)
    tensors = {}
    for name in INVENTORY:
        shp = shapes[name]
        if len(shp) == 1:
            raw = normal(seed, "norm:" + name, shp, std=norm_std, dtype="f32")
            if not raw_hf:
                raw = (raw.astype(np.float64) + 1.0).astype(np.float32)
            arr = to_bf16(raw) if s.dtype == "bf16" else raw
        else:
            arr = normal(seed, "w:" + name, shp, std=weight_std, dtype=s.dtype)
        tensors[("mtp." + name) if raw_hf else name] = arr
    embed = normal(seed, "embed_tokens", (s.vocab, s.hidden), std=weight_std, dtype=s.dtype)
    return Model(s, tensors, embed, raw_hf)


def kv_prefill(s: Shape, seed: int, rows: int, capacity: int, lengths, tag: str = "kv"):
    """Draft KV [rows][n_kv][capacity][head_dim] with slots < lengths[r] drawn N(0,1), rest 0."""
    shp = (rows, s.n_kv, capacity, s.head_dim)
    k = normal(seed, tag + ":k", shp, dtype=s.dtype)
    v = normal(seed, tag + ":v", shp, dtype=s.dtype)
    for r in range(rows):
        k[r, :, lengths[r]:, :] = 0
        v[r, :, lengths[r]:, :] = 0
    return k, v


def plant_logits(base: np.ndarray, drafts, coins) -> np.ndarray:
    """Synthetic target rows for a verify block: row i (i < d) has its argmax
    moved onto draft x_{i+1} when coins[i] (logit = max + 1), and otherwise
    made to differ from it (logit = second - 1 when x_{i+1} was the argmax).
    Row d (the bonus row) is left as drawn."""
    out = np.array(base, dtype=np.float32, copy=True)
    for i, x in enumerate(drafts):
        row = out[i]
        top = np.argsort(-row.astype(np.float64), kind="stable")[:2]
        if coins[i]:
            row[x] = row[top[0]] + np.float32(1.0)
        elif top[0] == x:
            row[x] = row[top[1]] - np.float32(1.0)
    return out
