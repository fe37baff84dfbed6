"""Helpers shared by the GPU parity tests (moving data between torch and the oracle's
numpy arrays, and the tolerance checks).  No NVFP4 arithmetic lives here."""
import numpy as np
import torch

from oracle import formats as F


def u16(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> uint16 bit patterns (numpy, CPU)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def npy(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def rel_err_floor(got: np.ndarray, ref: np.ndarray, floor_frac: float = 1e-2):
    """max_i |got_i - ref_i| / max(|ref_i|, tau), tau = floor_frac * rms(ref); and the
    normwise error ||got - ref|| / ||ref||."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tau = floor_frac * np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    err = np.abs(got - ref) / np.maximum(np.abs(ref), tau)
    nw = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    return float(err.max()) if err.size else 0.0, float(nw)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |v| (subnormal spacing below 2^-126)."""
    a = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(a)
    return np.exp2(np.maximum(e - 1, -126) - 7.0)


def check_bf16_against(got_bits: np.ndarray, ref: np.ndarray, rel: float = 1e-3, floor_frac: float = 1e-2):
    """A BF16 result against a float64 reference: within one BF16 ulp of the reference
    plus the float32-accumulation allowance rel * max(|ref|, tau)."""
    got = F.bf16_to_f32(got_bits).astype(np.float64)
    ref = np.asarray(ref, np.float64)
    tau = floor_frac * np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    bound = bf16_ulp(ref) + rel * np.maximum(np.abs(ref), tau)
    bad = np.abs(got - ref) > bound
    return int(bad.sum()), float((np.abs(got - ref) / np.maximum(bound, 1e-300)).max()) if ref.size else 0.0


def combine_violations(out_bits: np.ndarray, y_bits: np.ndarray, inv: np.ndarray, w: np.ndarray) -> int:
    """The weighted un-permute out[t] = BF16(sum_j fl32(w[t,j] * y[inv[t,j]])), summed in
    float32 in order j, against the exact float64 sum of the same BF16 y: each float32
    product and sum adds at most 2^-24 of sum_j |w y| (k products, k - 1 sums, then the
    BF16 rounding of the float32 total: half a BF16 ulp of a value that is itself within
    that bound).  Returns the number of elements of out outside the bound."""
    k = inv.shape[1]
    yv = F.bf16_to_f32(y_bits).astype(np.float64)
    wv = np.asarray(w, np.float32).astype(np.float64)
    mag = sum(np.abs(wv[:, j:j + 1] * yv[inv[:, j]]) for j in range(k))
    exact = sum(wv[:, j:j + 1] * yv[inv[:, j]] for j in range(k))
    got = F.bf16_to_f32(out_bits).astype(np.float64)
    slack = (k + 1) * 2.0 ** -24 * mag
    bound = 0.5 * np.exp2(np.frexp(np.abs(exact) + slack)[1] - 8.0) + slack
    return int(np.sum(np.abs(got - exact) > bound))


# --------------------------------------------------------------------------- GEMM-tiled layout
# Host implementation of the layout documented in include/nvfp4moe.h (blocks of R rows x
# 256 K-values: R*128 bytes of 128-byte-swizzled codes, then (R/128)*2048 bytes of scales).

def _tiled_index(rows_pad, K, R):
    kb = K // 256
    r = np.arange(rows_pad)[:, None]
    b = np.arange(K // 2)[None, :]
    blk, rr = r // R, r % R
    code_off = (blk * kb + b // 128) * (R * 144) + rr * 128 + (((b % 128) // 16) ^ (rr % 8)) * 16 + (b % 16)
    c = np.arange(K // 16)[None, :]
    cc = c % 16
    sf_off = ((blk * kb + c // 16) * (R * 144) + R * 128 + (rr // 128) * 2048 + (cc // 4) * 512
              + (rr % 128 % 32) * 16 + (rr % 128 // 32) * 4 + cc % 4)
    return code_off, sf_off


def pack_tiled_host(codes_nib: np.ndarray, sf_rowmajor: np.ndarray, R: int) -> np.ndarray:
    """codes nibbles [rows, K] + row-major scales [rows, K/16] -> tiled bytes (pad rows 0)."""
    rows, K = codes_nib.shape
    rows_pad = (rows + R - 1) // R * R
    out = np.zeros(rows_pad // R * (K // 256) * R * 144, np.uint8)
    co, so = _tiled_index(rows_pad, K, R)
    packed = F.pack_e2m1(codes_nib)
    out[co[:rows]] = packed
    out[so[:rows]] = sf_rowmajor
    return out


def untile_host(buf: np.ndarray, rows: int, K: int, R: int):
    """tiled bytes -> (codes nibbles [rows, K], row-major scales [rows, K/16])."""
    rows_pad = (rows + R - 1) // R * R
    co, so = _tiled_index(rows_pad, K, R)
    buf = np.asarray(buf, np.uint8)
    return F.unpack_e2m1(buf[co[:rows]]), buf[so[:rows]]
