"""Acceptance checks of CUDA outputs against the fp64 oracle (test helper).

gelu_and_mul_sparse, per element (ref = oracle's unrounded fp64 value):
  * |out - ref| <= 1e-2 |ref| + 2e-3;
  * the zero pattern: out != 0 exactly where g > cutoff (and the product is
    not zero), except inside the flip band |g - cutoff| < 1e-3 std, where
    either outcome is correct: out == 0, or the small value that the kernel's
    own fp32 cutoff gives, bounded by gelu(s) <= s with s < 2e-3 std;
  * NaN exactly where the oracle has NaN.
Rows with std == 0 have an empty band, so their zero pattern must match
exactly.

silu_and_mul: the bf16 output is within one ulp of the oracle's correctly
rounded bf16, the distance taken on the ordered integer line of bf16
patterns (+0 and -0 equal).
"""
from __future__ import annotations

import numpy as np
import torch

RTOL, ATOL, BAND = 1e-2, 2e-3, 1e-3


def bits_of(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu").contiguous()
    assert t.dtype == torch.bfloat16
    return t.view(torch.int16).numpy().view(np.uint16)


def f64_of_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# Per-element tolerance (rtol, atol) and the magnitude below which a value
# rounds to zero in the output type (half its smallest subnormal), by type.
# bf16 is the target specification's bound; fp16 and fp32 follow from their
# rounding (2^-11, 2^-24) plus the fp32 arithmetic of the kernels (tanh
# approximation 2^-12 for fp16, an accurate tanh for fp32; the fp32 cutoff
# error of ~1e-6 std times |u| sets atol).
TOLERANCES = {
    torch.bfloat16: (RTOL, ATOL, 2.0 ** -134),
    torch.float16: (1e-3, 1e-5, 2.0 ** -25),
    torch.float32: (1e-5, 1e-5, 2.0 ** -150),
}


def f64_of(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16/fp16/fp32 tensor (on any device)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def check_gelu(out: torch.Tensor, x: torch.Tensor, d: int, res, label: str = "") -> dict:
    """Assert the acceptance criteria; return summary statistics."""
    rtol, atol, tiny = TOLERANCES[out.dtype]
    y = f64_of(out)
    xf = f64_of(x)
    g = xf[:, :d]
    u = xf[:, d:2 * d]
    ref = res.ref
    assert y.shape == ref.shape, (label, y.shape, ref.shape)
    cutoff = res.cutoff[:, None]
    std = res.std[:, None]

    nan_ref = np.isnan(ref)
    nan_y = np.isnan(y)
    assert np.array_equal(nan_ref, nan_y), f"{label}: NaN pattern differs ({(nan_ref != nan_y).sum()} elements)"
    fin = ~nan_ref

    with np.errstate(invalid="ignore"):
        err = np.abs(y - ref)
        tol = rtol * np.abs(ref) + atol
        band = np.abs(g - cutoff) < BAND * std
        ok_val = err <= tol
        flip_bound = (2 * BAND * std) * np.abs(u) * 1.01 + atol
        ok_band = band & ((y == 0) | (np.abs(y) <= flip_bound) | ok_val)
        bad = fin & ~(ok_val | ok_band)
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(
            f"{label}: {bad.sum()} elements out of tolerance; first at ({r},{c}): "
            f"out={y[r, c]!r} ref={ref[r, c]!r} g={g[r, c]!r} u={u[r, c]!r} "
            f"cutoff={res.cutoff[r]!r} std={res.std[r]!r}")

    expect_nz = res.mask & (np.abs(ref) >= tiny)
    mism = fin & ~band & ((y != 0) != expect_nz)
    if mism.any():
        r, c = np.argwhere(mism)[0]
        raise AssertionError(
            f"{label}: {mism.sum()} zero-mask mismatches outside the flip band; first at "
            f"({r},{c}): out={y[r, c]!r} ref={ref[r, c]!r} g={g[r, c]!r} cutoff={res.cutoff[r]!r}")
    flips = int((fin & band & ((y != 0) != expect_nz)).sum())
    rel = np.where(fin & (np.abs(ref) > 1e-3), err / np.maximum(np.abs(ref), 1e-300), 0.0)
    return {"max_abs_err": float(np.nanmax(np.where(fin, err, 0.0))) if y.size else 0.0,
            "max_rel_err": float(rel.max()) if y.size else 0.0,
            "band_flips": flips, "zero_fraction": float((y == 0).mean()) if y.size else 0.0}


def ordered(bits: np.ndarray) -> np.ndarray:
    """bf16 patterns -> integers ordered like the values (+0 and -0 both 0)."""
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_silu(out: torch.Tensor, ref16: np.ndarray, label: str = "") -> int:
    """Assert <= 1 bf16 ulp from the correctly rounded oracle; return the max distance."""
    ob = bits_of(out)
    assert ob.shape == ref16.shape
    nan_o = (ob & 0x7FFF) > 0x7F80
    nan_r = (ref16 & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_o, nan_r), f"{label}: NaN pattern differs"
    dist = np.abs(ordered(ob) - ordered(ref16))[~nan_r]
    mx = int(dist.max()) if dist.size else 0
    assert mx <= 1, f"{label}: {int((dist > 1).sum())} elements more than 1 ulp away (max {mx})"
    return mx


def ulp_of(c: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of the element type at |c| (bf16: 8 significant bits, fp16: 11)."""
    if dtype == torch.float16:
        return np.spacing(np.abs(c).astype(np.float16)).astype(np.float64)
    return np.spacing(np.abs(c).astype(np.float32)).astype(np.float64) * 2.0 ** 16


def _row_native_failures(y, yb, rb, g, c, nan, expect_nz, dt):
    """Per-row check of one row against a reference: (zero-pattern mismatches
    away from the cutoff c, outputs more than one ulp away, flips)."""
    near = np.abs(g - c) <= ulp_of(np.array([c]), dt)[0]
    flips = ~nan & ((y != 0) != expect_nz)
    dist = np.abs(ordered(yb) - ordered(rb))
    return int((flips & ~near).sum()), int((~nan & ~flips & (dist > 1)).sum()), flips


def _adjacent(v: float, dt: torch.dtype, side: int) -> float:
    """The element-type value next to v (itself of that type) on `side` (+1 up, -1 down)."""
    b = int(torch.tensor([v], dtype=dt).view(torch.int16).numpy().view(np.uint16)[0])
    o = int(ordered(np.array([b], dtype=np.uint16))[0]) + side
    nb = o if o >= 0 else (0x8000 | -o)
    return float(torch.from_numpy(np.array([nb], dtype=np.uint16).view(np.int16)).view(dt)
                 .to(torch.float64)[0])


def _stat_roundings(v64: float, tol: float, dt: torch.dtype) -> list[float]:
    """The element-type values a statistic computed in fp32 may round to: the
    rounding of the exact value v64 (through fp32, as the oracle rounds), and
    its neighbour across the midpoint when v64 lies within tol of it."""
    r = float(torch.tensor(v64, dtype=torch.float64).to(torch.float32).to(dt).to(torch.float64))
    if v64 == r or not np.isfinite(v64):
        return [r]
    other = _adjacent(r, dt, 1 if v64 > r else -1)
    return [r, other] if abs(v64 - 0.5 * (r + other)) <= tol else [r]


def check_native(out: torch.Tensor, x: torch.Tensor, d: int, ref: np.ndarray, mask: np.ndarray,
                 cut: np.ndarray, label: str = "", z: float | None = None) -> dict:
    """Native-rounding acceptance: outside one rounding step of the row's cutoff
    the zero pattern equals {g > c} exactly; every output is within one
    element-type ulp of the (already rounded) oracle value.

    Several results are correct on a row whose exact mean or population std
    lies within the fp32 rounding-error bound of recursive summation
    (2^-24 sum|g| for the mean, 2^-24 (d/2 + 2) std for the std) of a midpoint
    between two element-type values: the kernel's fp32 statistic may round to
    either.  Given z, such a row also passes when it meets the same criteria
    against PyTorch's CPU composition of the native ops with the other
    rounding (the composition the native oracle reproduces bit for bit)."""
    import torch.nn.functional as F
    dt = out.dtype
    y = f64_of(out)
    xf = f64_of(x)
    g, u = xf[:, :d], xf[:, d:2 * d]
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan), f"{label}: NaN pattern differs"
    yb = out.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    rb = torch.from_numpy(ref).to(dt).view(torch.int16).numpy().view(np.uint16)
    expect_nz = mask & (ref != 0)
    n_flips, n_ulp1, n_alt = 0, 0, 0
    first_bad = None
    for r in range(y.shape[0]):
        away, far, flips = _row_native_failures(y[r], yb[r], rb[r], g[r], cut[r], nan[r],
                                                expect_nz[r], dt)
        if away == 0 and far == 0:
            n_flips += int(flips.sum())
            continue
        ok = False
        if z is not None and np.isfinite(g[r]).all():
            m64 = float(g[r].mean())
            s64 = float(np.sqrt(((g[r] - m64) ** 2).mean()))
            ms = _stat_roundings(m64, 2.0 ** -24 * float(np.abs(g[r]).sum()), dt)
            ss = _stat_roundings(s64, 2.0 ** -24 * (d / 2 + 2) * s64, dt)
            gt = x[r, :d].detach().cpu()
            ut = x[r, d:2 * d].detach().cpu()
            for mv in ms:
                for sv in ss:
                    if (mv, sv) == (ms[0], ss[0]):
                        continue
                    ct = torch.tensor(mv, dtype=dt) + torch.tensor(sv, dtype=dt) * z
                    alt = F.gelu(torch.relu(gt - ct), approximate="tanh") * ut
                    c_alt = float(ct.to(torch.float64))
                    ab = alt.contiguous().view(torch.int16).numpy().view(np.uint16)
                    a64 = alt.to(torch.float64).numpy()
                    a_away, a_far, a_flips = _row_native_failures(
                        y[r], yb[r], ab, g[r], c_alt, np.isnan(a64), (g[r] > c_alt) & (a64 != 0),
                        dt)
                    if a_away == 0 and a_far == 0:
                        ok = True
                        n_flips += int(a_flips.sum())
                        break
                if ok:
                    break
        if ok:
            n_alt += 1
            continue
        if first_bad is None:
            first_bad = (r, away, far)
    if first_bad is not None:
        r, away, far = first_bad
        if away:
            raise AssertionError(f"{label}: row {r}: {away} zero-pattern mismatches away from c")
        dist = np.abs(ordered(yb[r]) - ordered(rb[r]))
        c = int(np.argmax(dist))
        raise AssertionError(f"{label}: row {r}: {far} outputs more than 1 ulp away; first "
                             f"({r},{c}) out={y[r, c]!r} ref={ref[r, c]!r}")
    n_ulp1 = int((~nan & (np.abs(ordered(yb) - ordered(rb)) == 1)).sum())
    return {"flips_near_cutoff": n_flips, "ulp1": n_ulp1, "rows_other_rounding": n_alt}
