"""Shared helpers for the tests: host<->device transfers of exact bits and the
comparison metrics (the tolerances themselves are written in each test)."""
import numpy as np


def dev_u16(a: np.ndarray):
    """Upload uint16 words (bf16/fp16 bits) as a CUDA int16 tensor, same bits."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).cuda()


def dev_f16(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16).copy()).cuda()


def dev_f32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32).copy()).cuda()


def host_u16(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_ordered(bits: np.ndarray) -> np.ndarray:
    """Map fp16 words to integers whose differences count ulps (+0 and -0 both 0)."""
    u = bits.astype(np.int64)
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


def f16_ulp_distance(gpu_bits: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """ulps between fp16 results and an fp64 reference rounded to fp16 (ties to even)."""
    ref_bits = ref.astype(np.float16).view(np.uint16)
    return np.abs(f16_ordered(gpu_bits) - f16_ordered(ref_bits))


def conv_sample_points(N, Ho, Wo, C_out, n_random, seed=0) -> np.ndarray:
    """Flat NHWC output indices covering every border class (corners, edges,
    interior), the first and last channel and the last output row, plus random."""
    rng = np.random.default_rng(seed)
    hs = sorted({0, 1, Ho // 2, Ho - 2, Ho - 1} & set(range(Ho)))
    ws = sorted({0, 1, Wo // 2, Wo - 2, Wo - 1} & set(range(Wo)))
    cs = sorted({0, 1, C_out // 2, C_out - 1} & set(range(C_out)))
    pts = []
    for n in sorted({0, N - 1}):
        for h in hs:
            for w in ws:
                for c in cs:
                    pts.append(((n * Ho + h) * Wo + w) * C_out + c)
    total = N * Ho * Wo * C_out
    pts.extend(rng.integers(0, total, n_random).tolist())
    pts.extend(range(total - C_out, total))
    return np.unique(np.array(pts, np.int64))
