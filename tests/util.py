"""Shared helpers of the tests: bf16 views, tolerances and the teacher-forced step comparison."""
import numpy as np

# Tolerances on logits between the CUDA path (fp32 accumulation) and the fp64 oracle, as the
# benchmark's acceptance bar states them.
LOGIT_MAX_ABS = 2e-2
LOGIT_REL_L2 = 5e-3
ARGMAX_MARGIN = 5e-2


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """Round-to-nearest-even float32 -> bf16 bits (numpy, for building test inputs)."""
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def compare_logits(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    srt = np.sort(ref)
    margin = float(srt[-1] - srt[-2])
    return err, rel, margin


def ulp_diff_bf16(a, b):
    """Distance in bf16 steps between two arrays of bf16 bit patterns (same sign assumed)."""
    a = np.asarray(a, np.uint16).astype(np.int32)
    b = np.asarray(b, np.uint16).astype(np.int32)
    # map sign-magnitude to a monotone integer line
    ma = np.where(a & 0x8000, -(a & 0x7FFF), a & 0x7FFF)
    mb = np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(ma - mb)


def kv_close(gpu_bits, ref_bits, rel_floor=2e-4):
    """KV values written by the GPU (fp32 arithmetic, rounded to bf16) against the oracle's (fp64,
    rounded to bf16): equal up to one bf16 step at that magnitude, plus an absolute floor of
    rel_floor x the RMS of the reference values. The floor covers values near zero, where the fp32
    error carried by the residual stream and a long dot product exceeds a bf16 step; a wrong
    rotation, sign or slot errs by O(RMS) and still fails. Returns the worst excess (<= 0 when every
    value is close)."""
    a = bf16_to_f64(gpu_bits)
    b = bf16_to_f64(ref_bits)
    floor = rel_floor * float(np.sqrt(np.mean(b * b)))
    tol = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7 + floor
    return float((np.abs(a - b) - tol).max())


def kv_deviation(gpu_bits, ref_bits):
    """How GPU-written KV values (fp32 arithmetic, rounded to bf16) differ from the oracle's (fp64,
    rounded to bf16): the largest deviation in bf16 steps among values of magnitude at least 1/16 of
    the reference RMS, and the largest absolute deviation of the smaller values in multiples of that
    RMS (near zero a bf16 step is tiny, and the fp32 error carried by the residual stream and the
    dot product is what remains)."""
    a = bf16_to_f64(gpu_bits)
    b = bf16_to_f64(ref_bits)
    d = np.abs(a - b)
    rms = float(np.sqrt(np.mean(b * b)))
    big = np.abs(b) >= rms / 16
    step = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7
    steps_big = float((d[big] / step[big]).max()) if big.any() else 0.0
    small_rms = float(d[~big].max() / rms) if (~big).any() and rms > 0 else 0.0
    return steps_big, small_rms
