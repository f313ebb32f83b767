"""Helpers for comparing the CUDA path with the fp64 oracle.

Tolerances (what the hot path must meet against the fp64 recurrence):
  * fp32 q/k/v: relative L2 error <= 1e-4 on the output and on the final state;
  * bf16 q/k/v with fp32 state: relative L2 <= 1e-2 and max |err| <= 2e-2 * RMS
    of the reference, on the output and on the final state.
relative L2 = ||x - ref||_2 / ||ref||_2 over the whole compared tensor.

The max-error bound measures the computation, not the storage type: a bf16
output cannot hold the fp64 value closer than half a bf16 ulp of that value,
so that representation error (|ref| * 2^-9 at most) is discounted element by
element before the bound is applied.  Without the discount the rounding of
the largest outputs alone (|o| up to ~12 RMS on these workloads) exceeds
2e-2 * RMS even for an exact computation.
"""
import numpy as np
import torch

import oracle

TOL_F32 = 1e-4
TOL_BF16_REL = 1e-2
TOL_BF16_MAX_RMS = 2e-2


def as64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_l2(x, ref):
    x, ref = as64(x), as64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x))


def half_ulp(ref, dtype):
    """Half a unit in the last place of each value in `dtype` (bf16: 8
    significant bits, so half an ulp of |r| in [2^(E-1), 2^E) is 2^(E-9))."""
    ref = np.abs(as64(ref))
    if dtype != torch.bfloat16:
        return np.zeros_like(ref)
    _, e = np.frexp(ref)
    return np.where(ref > 0, np.ldexp(1.0, e - 9), 0.0)


def max_over_rms(x, ref, storage=None, roundings=1):
    x, ref = as64(x), as64(ref)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    err = np.abs(x - ref)
    if storage is not None:
        err = np.maximum(err - roundings * half_ulp(ref, storage), 0.0)
    return float(np.max(err, initial=0.0) / rms) if rms > 0 else float(np.max(err, initial=0.0))


def assert_close(x, ref, io_dtype, what="", both_stored=False):
    """The tolerance rule above, by io dtype (x's own dtype sets the storage
    rounding that is discounted).  both_stored: ref is itself a bf16 result
    of the library (two GPU paths compared), so each side carries its own
    half-ulp output rounding."""
    e = rel_l2(x, ref)
    if io_dtype == torch.float32:
        assert e <= TOL_F32, f"{what}: rel-L2 {e:.3e} > {TOL_F32}"
    else:
        storage = x.dtype if isinstance(x, torch.Tensor) else None
        m = max_over_rms(x, ref, storage, 2 if both_stored else 1)
        assert e <= TOL_BF16_REL, f"{what}: rel-L2 {e:.3e} > {TOL_BF16_REL}"
        assert m <= TOL_BF16_MAX_RMS, f"{what}: max|err|/RMS {m:.3e} > {TOL_BF16_MAX_RMS}"
    return e


def oracle_pairs(p, pairs, threads=0):
    """Run the oracle on selected (sequence, head) pairs of Problem p.
    Returns {(n, h): (out [L, dv], final [dk, dv])} in float64."""
    cu = p.cu_seqlens_host
    qs, ks, vs, zs, bs, s0s, lens = [], [], [], [], [], [], []
    for n, h in pairs:
        a, b = cu[n], cu[n + 1]
        qs.append(p.q[a:b, h:h + 1].cpu())
        ks.append(p.k[a:b, h:h + 1].cpu())
        vs.append(p.v[a:b, h:h + 1].cpu())
        zs.append(p.z[a:b, h:h + 1].cpu())
        bs.append(p.beta[a:b, h:h + 1].cpu())
        if p.initial_state is not None:
            s0s.append(p.initial_state[n:n + 1, h:h + 1].cpu())
        lens.append(b - a)
    cat = lambda xs: torch.cat(xs, 0)
    cu2 = np.concatenate([[0], np.cumsum(lens)])
    s0 = cat(s0s).reshape(len(pairs), 1, *s0s[0].shape[2:]) if s0s else None
    out, fin, _ = oracle.recurrent(cat(qs), cat(ks), cat(vs), cat(zs), cat(bs), cu2, s0,
                                   threads=threads)
    res = {}
    for i, (n, h) in enumerate(pairs):
        res[(n, h)] = (out[cu2[i]:cu2[i + 1], 0], fin[i, 0])
    return res
