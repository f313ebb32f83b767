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


class WholeTensorError:
    """Error statistics of one whole tensor, accumulated piece by piece.

    The tensor has a head axis (axis `head_axis` of every piece added); the
    sums of squared error and of squared reference values are kept per head,
    so that both the whole-tensor relative L2 error and the worst per-head
    value come out at the end, as do max |err| (after the storage half-ulp
    discount) and the whole-tensor RMS of the reference."""

    def __init__(self, num_heads, storage=None, roundings=1):
        self.err2 = np.zeros(num_heads)
        self.ref2 = np.zeros(num_heads)
        self.max_err = 0.0
        self.count = 0
        self.storage = storage
        self.roundings = roundings

    def add(self, x, ref, head_axis, heads=None):
        """x, ref: the same piece of the result and of the oracle; `heads` the
        head indices the piece's head axis holds (default: all of them)."""
        x, ref = as64(x), as64(ref)
        assert x.shape == ref.shape, (x.shape, ref.shape)
        d = x - ref
        axes = tuple(i for i in range(x.ndim) if i != head_axis)
        idx = np.arange(self.err2.size) if heads is None else np.asarray(heads)
        self.err2[idx] += np.sum(d * d, axis=axes)
        self.ref2[idx] += np.sum(ref * ref, axis=axes)
        err = np.abs(d)
        if self.storage is not None:
            err = np.maximum(err - self.roundings * half_ulp(ref, self.storage), 0.0)
        self.max_err = max(self.max_err, float(np.max(err, initial=0.0)))
        self.count += ref.size

    def rel_l2(self):
        den = float(np.sum(self.ref2))
        return float(np.sqrt(np.sum(self.err2) / den)) if den > 0 else float(np.sqrt(np.sum(self.err2)))

    def worst_head(self):
        with np.errstate(divide="ignore", invalid="ignore"):
            per = np.where(self.ref2 > 0, np.sqrt(self.err2 / self.ref2), np.sqrt(self.err2))
        h = int(np.argmax(per))
        return h, float(per[h])

    def max_over_rms(self):
        rms = np.sqrt(np.sum(self.ref2) / self.count) if self.count else 0.0
        return self.max_err / rms if rms > 0 else self.max_err

    def report(self, what):
        h, w = self.worst_head()
        return (f"{what}: rel-L2 {self.rel_l2():.3e} (worst head {h}: {w:.3e}), "
                f"max|err|/RMS {self.max_over_rms():.3e}")

    def check(self, io_dtype, what):
        """The tolerance rule of assert_close on the whole tensor."""
        e = self.rel_l2()
        if io_dtype == torch.float32:
            assert e <= TOL_F32, self.report(what)
        else:
            assert e <= TOL_BF16_REL, self.report(what)
            assert self.max_over_rms() <= TOL_BF16_MAX_RMS, self.report(what)
        return self.report(what)


def device_compare(x, ref, both_stored=False):
    """(rel-L2, max|err|/RMS) of two same-shape device tensors, computed in
    fp64 on their device (for comparisons too large to move to the host).
    both_stored: each side is a bf16 result, so two half-ulps are discounted."""
    xd, rd = x.double(), ref.double()
    d = xd - rd
    den = torch.linalg.vector_norm(rd)
    rel = float(torch.linalg.vector_norm(d) / den) if float(den) > 0 else float(
        torch.linalg.vector_norm(d))
    err = d.abs()
    if ref.dtype == torch.bfloat16 or x.dtype == torch.bfloat16:
        a = rd.abs()
        _, e = torch.frexp(a)
        hu = torch.where(a > 0, torch.ldexp(torch.ones_like(a), (e - 9).to(a.dtype)),
                         torch.zeros_like(a))
        err = torch.clamp(err - (2 if both_stored else 1) * hu, min=0.0)
    rms = torch.sqrt(torch.mean(rd * rd))
    mx = float(err.max()) if err.numel() else 0.0
    return rel, (mx / float(rms) if float(rms) > 0 else mx)


def problem_pieces(p, max_head_tokens=1 << 21):
    """(sequence range, head range) pieces covering a packed Problem p, each
    about max_head_tokens head-tokens of oracle work: groups of whole
    sequences, or groups of heads of a single sequence."""
    cu, H = p.cu_seqlens_host, p.meta["num_heads"]
    if p.num_seqs == 1:
        hs = max(1, min(H, max_head_tokens // max(cu[1], 1)))
        return [((0, 1), (h, min(H, h + hs))) for h in range(0, H, hs)]
    out, n0, tok = [], 0, 0
    for n in range(p.num_seqs):
        tok += (cu[n + 1] - cu[n]) * H
        if tok >= max_head_tokens or n + 1 == p.num_seqs:
            out.append(((n0, n + 1), (0, H)))
            n0, tok = n + 1, 0
    return out
