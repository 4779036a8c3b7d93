"""Seeded synthetic inputs shared by the oracle tests, the CUDA path's tests and the bench.

This module draws random numbers and quantises them to the storage type the GPU reads
(bf16, round-to-nearest-even).  It holds none of the method's arithmetic: no packing rule,
no embedding, no attention, no loss.  Both the oracle and the CUDA path consume exactly the
arrays produced here, so a disagreement between them is never an input mismatch.

Every tensor is drawn from its own counter-based stream, keyed by (seed, name, chunk), so
adding a tensor never shifts another one and the result does not depend on the number of
threads used to draw it.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 22


def _key(name: str) -> int:
    return zlib.crc32(name.encode("utf-8"))


def normal(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) of `shape`, drawn in fixed-size chunks (thread-count independent)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    chunks = [(i, min(n, i + _CHUNK)) for i in range(0, n, _CHUNK)]

    def fill(ci):
        lo, hi = chunks[ci]
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _key(name), ci])))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if len(chunks) > 2:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(len(chunks))))
    else:
        for ci in range(len(chunks)):
            fill(ci)
    return out.reshape(shape)


def rng(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _key(name)])))


# ---------------------------------------------------------------- bf16 storage quantisation
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values exactly representable in bf16 (the values the GPU sees)."""
    return bf16_bits_to_f32(f32_to_bf16_bits(a))


# ---------------------------------------------------------------- dims and samples
@dataclass(frozen=True)
class Dims:
    hidden: int        # H
    heads: int         # nh
    channels: int      # C, latent channels per patch token
    mlp_ratio: int = 4
    freq_dim: int = 256

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads


TINY = Dims(hidden=256, heads=4, channels=64)
FULL = Dims(hidden=3072, heads=24, channels=128)


@dataclass(frozen=True)
class Sample:
    """One packing candidate: text length, frame count and latent grid of one image."""
    txt_len: int
    frames: int
    lat_h: int
    lat_w: int
    t: float
    cfg_role: int = 0   # 0 plain, 1 cond, 2 uncond
    cfg_pair: int = -1  # index (in the candidate list) of the other branch

    @property
    def length(self) -> int:
        return self.txt_len + self.frames * self.lat_h * self.lat_w

    @property
    def img_len(self) -> int:
        return self.frames * self.lat_h * self.lat_w


def sample_array(samples) -> np.ndarray:
    """Samples as the packed struct array the C ABI reads (mf_sample, 28 bytes each)."""
    dt = np.dtype([("txt_len", "<i4"), ("frames", "<i4"), ("lat_h", "<i4"), ("lat_w", "<i4"),
                   ("t", "<f4"), ("cfg_role", "<i4"), ("cfg_pair", "<i4")])
    a = np.zeros(len(samples), dtype=dt)
    for i, s in enumerate(samples):
        a[i] = (s.txt_len, s.frames, s.lat_h, s.lat_w, np.float32(s.t), s.cfg_role, s.cfg_pair)
    return a


# ---------------------------------------------------------------- workloads
def tiny_samples(seed: int = 0):
    g = rng(seed, "tiny.t")
    t = g.uniform(0.0, 1.0, size=2).astype(np.float32)
    return [Sample(16, 1, 8, 8, float(t[0])), Sample(16, 1, 4, 12, float(t[1]))]


def gen1024_samples():
    return [Sample(256, 1, 64, 64, 0.5)]


def native_candidates(seed: int, n: int = 64, lo: int = 512, hi: int = 2048, txt_lo: int = 32,
                      txt_hi: int = 512):
    """Candidates for the 16384-token native-resolution pack: H, W uniform over multiples of 16
    in [lo, hi] (latent grid H/16 x W/16), text length uniform in [txt_lo, txt_hi], and
    t = sigmoid(N(0, 1)) (logit-normal)."""
    g = rng(seed, "native.candidates")
    steps = (hi - lo) // 16 + 1
    hh = lo // 16 + g.integers(0, steps, size=n)
    ww = lo // 16 + g.integers(0, steps, size=n)
    tl = g.integers(txt_lo, txt_hi + 1, size=n)
    u = g.standard_normal(n)
    t = (1.0 / (1.0 + np.exp(-u))).astype(np.float32)
    return [Sample(int(tl[i]), 1, int(hh[i]), int(ww[i]), float(t[i])) for i in range(n)]


def cfg_samples():
    """Two prompts (1024x1024 and 768x1344) with cond (256 text tokens) and uncond (no text)
    branches, in the order cond0, uncond0, cond1, uncond1."""
    return [Sample(256, 1, 64, 64, 1.0, 1, 1), Sample(0, 1, 64, 64, 1.0, 2, 0),
            Sample(256, 1, 48, 84, 1.0, 1, 3), Sample(0, 1, 48, 84, 1.0, 2, 2)]


def edit_samples(seed: int = 0):
    g = rng(seed, "edit.t")
    u = g.standard_normal(2)
    t = (1.0 / (1.0 + np.exp(-u))).astype(np.float32)
    return [Sample(512, 2, 64, 64, float(t[0])), Sample(512, 2, 64, 64, float(t[1]))]


# ---------------------------------------------------------------- weights
# Weight matrices are stored [out_features][in_features] (row-major), biases [out_features].
BLOCK_SHAPES = lambda d: {                                            # noqa: E731
    "w_mod": (6 * d.hidden, d.hidden), "b_mod": (6 * d.hidden,),
    "w_qkv": (3 * d.hidden, d.hidden), "b_qkv": (3 * d.hidden,),
    "w_o": (d.hidden, d.hidden), "b_o": (d.hidden,),
    "w_1": (d.mlp_ratio * d.hidden, d.hidden), "b_1": (d.mlp_ratio * d.hidden,),
    "w_2": (d.hidden, d.mlp_ratio * d.hidden), "b_2": (d.hidden,),
}
STREAMS = ("txt", "img")


@dataclass
class ModelWeights:
    """All weights of an n-block stack as float32 arrays.  `bf16=True` means every value is
    exactly representable in bf16 (the values uploaded to the GPU)."""
    dims: Dims
    temb: dict = field(default_factory=dict)     # w_t1 [H][F], b_t1, w_t2 [H][H], b_t2
    embed: dict = field(default_factory=dict)    # w_in [H][C], b_in [H]
    blocks: list = field(default_factory=list)   # [ {stream: {name: array}} ]
    final: dict = field(default_factory=dict)    # w_fmod [2H][H], b_fmod, w_out [C][H], b_out
    bf16: bool = False

    def arrays(self):
        """(name, array) over every tensor, in a fixed order."""
        for k in sorted(self.temb):
            yield "temb." + k, self.temb[k]
        for k in sorted(self.embed):
            yield "embed." + k, self.embed[k]
        for i, b in enumerate(self.blocks):
            for s in STREAMS:
                for k in sorted(b[s]):
                    yield f"block{i}.{s}.{k}", b[s][k]
        for k in sorted(self.final):
            yield "final." + k, self.final[k]

    def rounded(self) -> "ModelWeights":
        m = ModelWeights(self.dims, {k: round_bf16(v) for k, v in self.temb.items()},
                         {k: round_bf16(v) for k, v in self.embed.items()},
                         [{s: {k: round_bf16(v) for k, v in b[s].items()} for s in STREAMS}
                          for b in self.blocks],
                         {k: round_bf16(v) for k, v in self.final.items()}, True)
        return m


def model_weights(dims: Dims, n_blocks: int, seed: int, std: float = 0.02,
                  bf16: bool = True, qk_norm: bool = False) -> ModelWeights:
    """Seeded weights of an n-block stack.  qk_norm adds the QK-RMSNorm scales of each stream
    (w_qnorm, w_knorm [head_dim], 1 + N(0, 0.1^2))."""
    d = dims
    H, C, F = d.hidden, d.channels, d.freq_dim
    nm = lambda name, shape: normal(seed, name, shape, std)            # noqa: E731
    m = ModelWeights(d)
    m.temb = {"w_t1": nm("temb.w_t1", (H, F)), "b_t1": nm("temb.b_t1", (H,)),
              "w_t2": nm("temb.w_t2", (H, H)), "b_t2": nm("temb.b_t2", (H,))}
    m.embed = {"w_in": nm("embed.w_in", (H, C)), "b_in": nm("embed.b_in", (H,))}
    for i in range(n_blocks):
        m.blocks.append({s: {k: nm(f"block{i}.{s}.{k}", shp) for k, shp in BLOCK_SHAPES(d).items()}
                         for s in STREAMS})
        if qk_norm:
            for s in STREAMS:
                for k in ("w_qnorm", "w_knorm"):
                    m.blocks[-1][s][k] = 1.0 + normal(seed, f"block{i}.{s}.{k}", (d.head_dim,), 0.1)
    m.final = {"w_fmod": nm("final.w_fmod", (2 * H, H)), "b_fmod": nm("final.b_fmod", (2 * H,)),
               "w_out": nm("final.w_out", (C, H)), "b_out": nm("final.b_out", (C,))}
    return m.rounded() if bf16 else m


# ---------------------------------------------------------------- activations
@dataclass
class Batch:
    """Per-candidate inputs.  x_txt[i]: [txt_len][H] text embeddings; z[i], eps[i]:
    [frames*h*w][C] clean latents and noise, frame-major then row-major."""
    samples: list
    x_txt: list
    z: list
    eps: list


def batch_inputs(samples, dims: Dims, seed: int, bf16: bool = True) -> Batch:
    H, C = dims.hidden, dims.channels
    xs, zs, es = [], [], []
    for i, s in enumerate(samples):
        x = normal(seed, f"x_txt.{i}", (s.txt_len, H))
        z = normal(seed, f"z.{i}", (s.img_len, C))
        e = normal(seed, f"eps.{i}", (s.img_len, C))
        if bf16:
            x, z, e = round_bf16(x), round_bf16(z), round_bf16(e)
        xs.append(x), zs.append(z), es.append(e)
    return Batch(list(samples), xs, zs, es)


def pack_inputs(samples, order, dims: Dims, seed: int):
    """Inputs of the packed candidates only, concatenated in stream order (pack order):
    x_txt [N_txt][H], z and eps [N_img][C], all bf16-exact float32.  Candidate c draws the same
    values as batch_inputs() gives it (the streams are keyed by candidate index)."""
    H, C = dims.hidden, dims.channels
    xs = [round_bf16(normal(seed, f"x_txt.{c}", (samples[c].txt_len, H))) for c in order]
    zs = [round_bf16(normal(seed, f"z.{c}", (samples[c].img_len, C))) for c in order]
    es = [round_bf16(normal(seed, f"eps.{c}", (samples[c].img_len, C))) for c in order]
    cat = lambda a, w: np.concatenate(a) if a else np.zeros((0, w), np.float32)   # noqa: E731
    return cat(xs, H), cat(zs, C), cat(es, C)


def cfg_batch(samples, dims: Dims, seed: int) -> Batch:
    """Packed-CFG inputs: each uncond branch shares its cond partner's starting noise z0
    (stored in `z`) and takes no text."""
    b = batch_inputs(samples, dims, seed)
    for i, s in enumerate(samples):
        if s.cfg_role == 2:
            b.z[i] = b.z[s.cfg_pair]
            b.eps[i] = b.eps[s.cfg_pair]
    return b
