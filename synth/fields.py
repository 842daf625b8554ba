"""Seeded synthetic stand-ins for Lorenzo-quantized climate residuals.

The GPULZ stage page measures on 24.7 MB of Lorenzo-quantized CESM CLDHGH
residuals (a 1800x3600 float32 field). That dataset is not available here, so
each workload is a synthetic field of the same shape and code distribution:

* field: sum of 8 seeded random sinusoids
  ``a_k * sin(2*pi*<d_k, x>/lambda_k + phi_k)`` over pixel coordinates, with
  ``lambda_k`` log-uniform in [8, 128] px, ``d_k`` a uniform random unit
  direction (2D for plane fields, 3D for volumes), ``phi_k ~ U[0, 2*pi)``,
  ``a_k ~ U[0.5, 1.5]``; plus Gaussian noise ``N(0, 1e-3 * range)`` where
  ``range`` is max - min of the noiseless sum. Computed in float64, stored as
  float32.
* quantization (pre-quantized Lorenzo, plain reading): absolute error bound
  ``eb = eb_rel * range`` of the noisy float32 field; ``q = round(x / (2 eb))``
  rounding half away from zero in float64; Lorenzo delta on the integer grid
  with zero outside (2D: 4-term, 3D: 8-term inclusion-exclusion; the byte
  workload applies 2D per z-slice); ``code = clamp(delta + R, 0, 2R - 1)``.
* layout: row-major, x fastest; volumes z-major.
* sparse workload (mostly-zero codes, the zero-chunk path at scale): the same
  2D field, quantized as ``q = round(max(x - t, 0) / (2 eb))`` with the
  threshold ``t`` at 90 % of the noisy field's range, stored as u16; only the
  sinusoid crests are nonzero (about 0.1 % of the codes; about 70 % of
  the 2 KB chunks are all zero).

Everything is deterministic in the seed (numpy PCG64).
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np


def _workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    shape: tuple            # (ny, nx) or (nz, ny, nx)
    directions: int         # 2 or 3 (dimension of the sinusoid directions)
    lorenzo: str            # "2d", "3d", "2d_per_slice" or "sparse"
    eb_rel: float
    radius: int
    dtype: str              # "u32", "u16" or "u8"
    chunk_size: int
    word_size: int
    match_level: int
    seed: int

    @property
    def n_bytes(self) -> int:
        return int(np.prod(self.shape)) * {"u32": 4, "u16": 2, "u8": 1}[self.dtype]

    @property
    def codes(self) -> str:
        if self.lorenzo == "sparse":
            return "thresholded crest codes (%s, 90%% of range)" % self.dtype
        return "%s Lorenzo codes (%s, radius %d)" % (self.lorenzo, self.dtype, self.radius)

    def describe(self) -> str:
        dims = "x".join(str(s) for s in self.shape)
        return ("%s %s float32 field -> %s, chunk_size=%d, word_size=%d, match_level=%d"
                % (self.name, dims, self.codes, self.chunk_size, self.word_size,
                   self.match_level))


# The workloads: a tiny plane, the 1800x3600 plane at both match levels,
# a 512^3 volume, the 1800x3600x16 byte stream, the plane as u16 codes and a
# mostly-zero u16 field.
CONFIGS = {
    1: Config("tiny_256x256_u32", (256, 256), 2, "2d", 1e-3, 32768, "u32", 2048, 4, 0,
              20261202 + 1),
    2: Config("plane_1800x3600_u32_l0", (1800, 3600), 2, "2d", 1e-3, 32768, "u32", 2048, 4, 0,
              20261202 + 2),
    3: Config("plane_1800x3600_u32_l1", (1800, 3600), 2, "2d", 1e-3, 32768, "u32", 2048, 4, 1,
              20261202 + 3),
    4: Config("volume_512cube_u32_l1", (512, 512, 512), 3, "3d", 1e-3, 32768, "u32", 4096, 4,
              1, 20261202 + 4),
    5: Config("bytes_1800x3600x16_u8_l1", (16, 1800, 3600), 3, "2d_per_slice", 1e-2, 128, "u8",
              4096, 1, 1, 20261202 + 5),
    # word_size 2 (u16 codes, the pages' common pairing with a 16-bit entropy
    # coder) and a mostly-zero input exercising zero chunks at scale
    6: Config("plane_1800x3600_u16_l1", (1800, 3600), 2, "2d", 1e-3, 32768, "u16", 4096, 2, 1,
              20261202 + 6),
    7: Config("sparse_4096x4096_u16_l0", (4096, 4096), 2, "sparse", 1e-3, 32768, "u16", 2048, 2,
              0, 20261202 + 7),
}


def _draw_terms(rng: np.random.Generator, directions: int):
    terms = []
    for _ in range(8):
        lam = math.exp(rng.uniform(math.log(8.0), math.log(128.0)))
        if directions == 2:
            ang = rng.uniform(0.0, 2.0 * math.pi)
            d = np.array([math.cos(ang), math.sin(ang)])
        else:
            v = rng.standard_normal(3)
            d = v / np.linalg.norm(v)
        phi = rng.uniform(0.0, 2.0 * math.pi)
        amp = rng.uniform(0.5, 1.5)
        terms.append((lam, d, phi, amp))
    return terms


def _plane_sum(terms, ny: int, nx: int, z: float | None) -> np.ndarray:
    """Noiseless sum of the sinusoids on one (ny, nx) plane (optionally at depth z)."""
    y = np.arange(ny, dtype=np.float64)[:, None]
    x = np.arange(nx, dtype=np.float64)[None, :]
    f = np.zeros((ny, nx), np.float64)
    for lam, d, phi, amp in terms:
        k = 2.0 * math.pi / lam
        if d.size == 2:
            arg = k * (d[0] * x + d[1] * y) + phi
        else:
            arg = k * (d[0] * x + d[1] * y + d[2] * (z or 0.0)) + phi
        f += amp * np.sin(arg)
    return f


def generate_field(cfg: Config, seed: int | None = None) -> np.ndarray:
    """The float32 field of a workload (noise included)."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    terms = _draw_terms(rng, cfg.directions)
    if len(cfg.shape) == 2:
        ny, nx = cfg.shape
        clean = _plane_sum(terms, ny, nx, None)
        rng_f = float(clean.max() - clean.min())
        noisy = clean + rng.normal(0.0, 1e-3 * rng_f, size=clean.shape)
        return noisy.astype(np.float32)
    nz, ny, nx = cfg.shape
    workers = _workers()

    def plane_at(z):
        return _plane_sum(terms, ny, nx, float(z))

    def extent(z):
        plane = plane_at(z)
        return float(plane.min()), float(plane.max())

    # the planes are independent (computed on host threads, in any order); the
    # noise is drawn in z order from the one generator, so the field does not
    # depend on the number of threads
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        ext = list(ex.map(extent, range(nz)))
        lo = min(e[0] for e in ext)
        hi = max(e[1] for e in ext)
        sigma = 1e-3 * (hi - lo)
        out = np.empty(cfg.shape, np.float32)
        for z0 in range(0, nz, workers):
            zs = range(z0, min(nz, z0 + workers))
            for z, plane in zip(zs, ex.map(plane_at, zs)):
                out[z] = (plane + rng.normal(0.0, sigma, size=plane.shape)).astype(np.float32)
    return out


def _round_half_away(v: np.ndarray) -> np.ndarray:
    return (np.sign(v) * np.floor(np.abs(v) + 0.5)).astype(np.int64)


def _lorenzo_2d(q: np.ndarray) -> np.ndarray:
    p = np.zeros((q.shape[0] + 1, q.shape[1] + 1), np.int64)
    p[1:, 1:] = q
    return p[1:, 1:] - p[:-1, 1:] - p[1:, :-1] + p[:-1, :-1]


def lorenzo_codes(field: np.ndarray, cfg: Config) -> np.ndarray:
    """Quantize + Lorenzo-predict a field into the workload's integer codes."""
    f64_lo = float(field.min())
    f64_hi = float(field.max())
    eb = cfg.eb_rel * (f64_hi - f64_lo)
    if eb <= 0.0:
        eb = 1.0
    dt = {"u32": np.uint32, "u16": np.uint16, "u8": np.uint8}[cfg.dtype]
    R = cfg.radius
    if cfg.lorenzo == "sparse":
        t = f64_lo + 0.90 * (f64_hi - f64_lo)
        q = _round_half_away(np.maximum(field.astype(np.float64) - t, 0.0) / (2.0 * eb))
        return np.clip(q, 0, 65535).astype(dt)
    if cfg.lorenzo == "2d":
        q = _round_half_away(field.astype(np.float64) / (2.0 * eb))
        delta = _lorenzo_2d(q)
        return np.clip(delta + R, 0, 2 * R - 1).astype(dt)
    out = np.empty(field.shape, dt)
    nz = field.shape[0]

    def quant(z):
        return _round_half_away(field[z].astype(np.float64) / (2.0 * eb))

    def slice_codes(z):
        # 3D: the 2D delta of slice z minus that of slice z - 1 (zero outside)
        d2 = _lorenzo_2d(quant(z))
        if cfg.lorenzo == "3d" and z > 0:
            d2 = d2 - _lorenzo_2d(quant(z - 1))
        out[z] = np.clip(d2 + R, 0, 2 * R - 1).astype(dt)

    with concurrent.futures.ThreadPoolExecutor(_workers()) as ex:
        list(ex.map(slice_codes, range(nz)))
    return out


def generate(cfg_id: int | Config, seed: int | None = None) -> np.ndarray:
    """Codes of a workload as a flat little-endian byte array (np.uint8)."""
    cfg = CONFIGS[cfg_id] if isinstance(cfg_id, int) else cfg_id
    codes = lorenzo_codes(generate_field(cfg, seed), cfg)
    return np.ascontiguousarray(codes).reshape(-1).view(np.uint8)
