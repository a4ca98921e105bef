"""Checks that pin the CPU oracle to facts fixed outside the oracle itself.

Each check takes an ``oracle.Oracle`` and returns a list of failure strings,
so the same checks run against the committed oracle (tests/test_oracle_pins.py,
which wants no failures) and against copies with planted mistakes
(tests/test_oracle_mutants.py, which wants at least one failure each).

What pins what:
  * bf16 rounding  -> torch's fp32->bf16 conversion (a library routine) and
                      hand-derived ties, subnormals and the overflow edge;
  * hand rows      -> tests/golden/hand_rows.json, values derived on paper;
  * brute force    -> exact rational arithmetic (fractions / decimal) on
                      dyadic inputs whose fp32 sums are exact;
  * error bound    -> the textbook bound of recursive fp32 summation;
  * n = 1          -> torch.nn.functional.rms_norm in float64 (library);
  * invariants     -> rms(out / w) ~ 1 and scaling by powers of two.
"""
import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_rows.json")

BF16_REL = 2.0 ** -7   # output tolerance: |err| <= 2^-7 |ref| + 1e-3
BF16_ABS = 1e-3


def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_to_bf16_bits_exact(values) -> np.ndarray:
    """Patterns of values that are already bf16-exact (checked)."""
    x = np.asarray(values, dtype=np.float32)
    b = torch_bf16_bits(x)
    back = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert np.array_equal(back, x), "fixture value is not bf16-exact"
    return b


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- bf16 rounding

def check_bf16_rounding_vs_torch(orc):
    fails = []
    rng = np.random.default_rng(1234)
    # magnitudes from deep subnormal to past the bf16 overflow edge
    mant = rng.uniform(1.0, 2.0, 4000).astype(np.float32)
    expo = rng.integers(-149, 128, 4000)
    x = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    x *= np.where(rng.random(4000) < 0.5, -1, 1).astype(np.float32)
    # exact ties, one below and one above, with even and odd kept bits
    base = rng.integers(0, 0x7F7F, 2000).astype(np.uint32) << 16
    ties = np.concatenate([base | 0x8000, base | 0x7FFF, base | 0x8001,
                           (base | 0x10000) | 0x8000]).astype(np.uint32)
    x = np.concatenate([x, ties.view(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38,
                                  3.3961776e38, 3.4028235e38], np.float32)])
    x = x[np.isfinite(x) | np.isinf(x)]
    want = torch_bf16_bits(x)
    got = orc.bf16_from_f64(x.astype(np.float64))
    bad = np.nonzero(want != got)[0]
    if bad.size:
        i = bad[0]
        fails.append(f"bf16 rounding of {x[i]!r}: oracle {got[i]:#06x}, torch {want[i]:#06x}"
                     f" ({bad.size} mismatches)")
    # widening is exact
    pats = np.arange(0, 1 << 16, 7, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7F80) != 0x7F80]   # skip inf/NaN patterns
    wide = orc.bf16_to_f32(pats)
    if not np.array_equal(wide.view(np.uint32), pats.astype(np.uint32) << 16):
        fails.append("bf16 -> fp32 widening is not the top-half placement")
    return fails


def check_bf16_rounding_by_hand(orc):
    """Single rounding straight from fp64, derived by hand."""
    cases = [
        (1 + 2 ** -8, 0x3F80),               # tie between 1 and 1+2^-7 -> even 1
        (1 + 3 * 2 ** -8, 0x3F82),           # tie between 1+2^-7 and 1+2^-6 -> even
        (1 + 2 ** -8 + 2 ** -40, 0x3F81),    # just above a tie: up (fp32-first would tie to 1)
        (-(1 + 2 ** -8 + 2 ** -40), 0xBF81),
        (2.0 ** -133, 0x0001),               # smallest subnormal
        (2.0 ** -134, 0x0000),               # tie between 0 and 2^-133 -> 0
        (1.5 * 2.0 ** -134, 0x0001),
        (3 * 2.0 ** -134, 0x0002),           # 1.5 quanta: tie -> even 2
        (2.0 ** -126, 0x0080),               # smallest normal
        (float.fromhex("0x1.FEp127"), 0x7F7F),   # largest finite: (2 - 2^-7) 2^127
        (float.fromhex("0x1.FE8p127"), 0x7F7F),  # below the overflow tie
        (float.fromhex("0x1.FFp127"), 0x7F80),   # the tie overflows (even) -> inf
        (-0.0, 0x8000),
        (0.1, 0x3DCD),                        # 0.1 = 1.6 * 2^-4 -> 1 + 77/128
    ]
    xs = np.array([c[0] for c in cases], dtype=np.float64)
    got = orc.bf16_from_f64(xs)
    return [f"bf16({c[0]!r}) = {g:#06x}, expected {c[1]:#06x}"
            for c, g in zip(cases, got) if int(g) != c[1]]


# ---------------------------------------------------------------- hand rows

def _as_rows(a):
    a = np.asarray(a, dtype=np.float32)
    return a.reshape(1, -1) if a.ndim == 1 else a


def check_hand_rows(orc):
    fails = []
    with open(GOLDEN) as f:
        rows = json.load(f)["rows"]
    for row in rows:
        parts = [f32_to_bf16_bits_exact(_as_rows(p)) for p in row["partials"]]
        res = f32_to_bf16_bits_exact(_as_rows(row["residual"]))
        w = f32_to_bf16_bits_exact(row["weight"])
        for mode in ("one_stage", "two_stage"):
            exp = row[mode]
            out, rout, s = orc.ar_rmsnorm(parts, res, w, row["eps"], two_stage=(mode == "two_stage"))
            tag = f"{row['name']}/{mode}"
            if not np.array_equal(s, _as_rows(exp["sum"])):
                fails.append(f"{tag}: sum {s.tolist()} != {exp['sum']}")
            if not np.array_equal(bits_to_f32(rout), _as_rows(exp["residual_out"])):
                fails.append(f"{tag}: residual_out {bits_to_f32(rout).tolist()} != {exp['residual_out']}")
            if "out_bits" in exp:
                want = np.array([int(b, 16) for b in exp["out_bits"]], dtype=np.uint16).reshape(out.shape)
                if not np.array_equal(out, want):
                    fails.append(f"{tag}: out {[hex(v) for v in out.ravel()]} != {exp['out_bits']}")
            else:
                if not np.array_equal(bits_to_f32(out), _as_rows(exp["out"])):
                    fails.append(f"{tag}: out {bits_to_f32(out).tolist()} != {exp['out']}")
    return fails


def check_tree_order_would_differ(orc):
    """n = 4: p = [16384, 0, 3*2^-12, 3*2^-12].

    In rank order every small term is below half the fp32 spacing at 16384
    (2^-10) and vanishes: the sum is 16384.  A pairwise tree would first add
    the two small terms (6*2^-12 = 1.5*2^-10 > 2^-10) and round up to
    16384 + 2^-9.
    """
    p = [np.full((1, 8), v, dtype=np.float32) for v in (16384.0, 0.0, 3 * 2 ** -12, 3 * 2 ** -12)]
    parts = [f32_to_bf16_bits_exact(x) for x in p]
    res = f32_to_bf16_bits_exact(np.zeros((1, 8), np.float32))
    w = f32_to_bf16_bits_exact(np.ones(8, np.float32))
    _, _, s = orc.ar_rmsnorm(parts, res, w, 1e-6)
    if not np.all(s == 16384.0):
        return [f"rank-order sum of [16384, 0, 3*2^-12, 3*2^-12] gave {s.ravel()[0]!r}, expected 16384"]
    return []


# ---------------------------------------------------------------- brute force

def bf16_rne_exact(q: Fraction) -> Fraction:
    """Nearest bf16 to an exact rational, ties to even (normal/subnormal range)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    quantum = Fraction(2) ** (max(e, -126) - 7)
    k = round(a / quantum)           # Fraction.__round__: half to even
    return sign * k * quantum


def check_brute_force_dyadic(orc, seed=7):
    """Dyadic inputs (multiples of 1/8 in [-8, 8]): every fp32 sum is exact,
    so sum and residual_out follow from exact rational arithmetic, and out
    from a 50-digit decimal square root."""
    fails = []
    getcontext().prec = 50
    rng = np.random.default_rng(seed)
    for n, m, H in [(1, 2, 8), (2, 3, 16), (3, 2, 24), (5, 2, 8), (8, 4, 32), (16, 2, 16)]:
        P = rng.integers(-64, 65, size=(n, m, H)) / 8.0
        R = rng.integers(-64, 65, size=(m, H)) / 8.0
        W = rng.integers(-16, 17, size=(H,)) / 8.0
        eps = float(np.float32(2.0 ** -10))
        parts = [f32_to_bf16_bits_exact(P[k]) for k in range(n)]
        res = f32_to_bf16_bits_exact(R)
        w = f32_to_bf16_bits_exact(W)
        for two in (False, True):
            out, rout, s = orc.ar_rmsnorm(parts, res, w, eps, two_stage=two)
            for i in range(m):
                rs = []
                for j in range(H):
                    acc = sum(Fraction(float(P[k, i, j])) for k in range(n))
                    if two:
                        acc = bf16_rne_exact(acc)
                    if Fraction(float(s[i, j])) != acc:
                        fails.append(f"brute n={n} two={two} sum[{i},{j}] {s[i, j]} != {float(acc)}")
                    r = acc + Fraction(float(R[i, j]))
                    rs.append(r)
                    if Fraction(float(bits_to_f32(rout[i, j]))) != bf16_rne_exact(r):
                        fails.append(f"brute n={n} two={two} residual_out[{i},{j}]")
                ss = sum(r * r for r in rs)
                inv = 1 / (Decimal(ss.numerator) / Decimal(ss.denominator) / H
                           + Decimal(eps)).sqrt()
                for j in range(H):
                    y = Decimal(rs[j].numerator) / Decimal(rs[j].denominator) * inv * Decimal(float(W[j]))
                    yq = Fraction(y)
                    want = bf16_rne_exact(yq)
                    got = Fraction(float(bits_to_f32(out[i, j])))
                    if got != want:
                        # allow only when y sits within 1e-12 (relative) of a rounding tie
                        lo = bf16_rne_exact(yq * (1 - Fraction(1, 10 ** 12)))
                        hi = bf16_rne_exact(yq * (1 + Fraction(1, 10 ** 12)))
                        if lo == hi:
                            fails.append(f"brute n={n} two={two} out[{i},{j}] {float(got)} != {float(want)}")
    return fails[:20]


# ---------------------------------------------------------------- bounds / invariants

def random_case(rng, n, m, H, p_std=0.5, r_std=1.0):
    P = [torch_bf16_bits(rng.normal(0, p_std, (m, H)).astype(np.float32)) for _ in range(n)]
    R = torch_bf16_bits(rng.normal(0, r_std, (m, H)).astype(np.float32))
    W = torch_bf16_bits(rng.normal(1, 0.1, (H,)).astype(np.float32))
    return P, R, W


def check_sum_error_bound(orc):
    """Recursive fp32 summation of n terms: |acc - S| <= gamma_{n-1} sum|p_k|,
    gamma_k = k u / (1 - k u), u = 2^-24 (a textbook bound)."""
    rng = np.random.default_rng(11)
    n, m, H = 8, 4, 512
    P, R, W = random_case(rng, n, m, H)
    # spread the magnitudes over 2^-12 .. 2^12 so that fp32 sums round often
    P = [torch_bf16_bits(bits_to_f32(p) * np.exp2(rng.integers(-12, 13, p.shape)).astype(np.float32))
         for p in P]
    _, _, s = orc.ar_rmsnorm(P, R, W, 1e-6)
    vals = np.stack([bits_to_f32(p).astype(np.float64) for p in P])
    exact = np.array([[math.fsum(vals[:, i, j]) for j in range(H)] for i in range(m)])
    u = 2.0 ** -24
    gamma = (n - 1) * u / (1 - (n - 1) * u)
    bound = gamma * np.abs(vals).sum(axis=0)
    err = np.abs(s.astype(np.float64) - exact)
    if np.any(err > bound):
        return [f"fp32 sum exceeds the recursive-summation bound by {float((err - bound).max())}"]
    return []


def check_n1_is_textbook_rmsnorm(orc):
    """n = 1: the sum is the partial itself, the two modes agree, and out is
    torch's fp64 rms_norm of (partial + residual), rounded to bf16."""
    fails = []
    rng = np.random.default_rng(5)
    m, H, eps = 6, 1024, 1e-6
    P, R, W = random_case(rng, 1, m, H)
    out1, rout1, s1 = orc.ar_rmsnorm(P, R, W, eps)
    out2, rout2, s2 = orc.ar_rmsnorm(P, R, W, eps, two_stage=True)
    if not (np.array_equal(out1, out2) and np.array_equal(rout1, rout2) and np.array_equal(s1, s2)):
        fails.append("n=1: one-stage and two-stage differ")
    if not np.array_equal(s1, bits_to_f32(P[0])):
        fails.append("n=1: the sum is not the partial")
    x = torch.from_numpy(bits_to_f32(P[0]).astype(np.float32)) + torch.from_numpy(bits_to_f32(R))
    y = torch.nn.functional.rms_norm(x.double(), (H,), torch.from_numpy(bits_to_f32(W)).double(),
                                     eps=float(np.float32(eps)))
    want = torch_bf16_bits(y.float().numpy())
    exact_frac = float(np.mean(want == out1))
    diff = np.abs(bits_to_f32(out1).astype(np.float64) - bits_to_f32(want))
    tol = BF16_REL * np.abs(bits_to_f32(want)) + BF16_ABS
    if exact_frac < 0.999 or np.any(diff > tol):
        fails.append(f"n=1: out vs torch rms_norm: {exact_frac:.5f} bit-equal, max diff {diff.max()}")
    if not np.array_equal(rout1, torch_bf16_bits(x.numpy())):
        fails.append("n=1: residual_out is not bf16(partial + residual)")
    return fails


def check_rms_invariant(orc):
    """rms_j(out_j / w_j) = sqrt(ms / (ms + eps)) up to bf16 rounding of out."""
    rng = np.random.default_rng(3)
    m, H, eps = 8, 2048, 1e-6
    P, R, W = random_case(rng, 4, m, H)
    out, rout, _ = orc.ar_rmsnorm(P, R, W, eps)
    y = bits_to_f32(out).astype(np.float64) / bits_to_f32(W).astype(np.float64)
    rms = np.sqrt(np.mean(y * y, axis=1))
    r = bits_to_f32(rout).astype(np.float64)
    ms = np.mean(r * r, axis=1)
    want = np.sqrt(ms / (ms + np.float32(eps)))
    if np.any(np.abs(rms - want) > 2.0 ** -8 * want):
        return [f"rms(out/w) off by {float(np.abs(rms - want).max())}"]
    return []


def check_scale_invariance(orc):
    """Scaling partials and residual by c = 2^k scales sum and residual_out
    exactly and leaves out unchanged (up to the eps term)."""
    fails = []
    rng = np.random.default_rng(9)
    m, H, eps = 4, 512, 1e-6
    P, R, W = random_case(rng, 8, m, H)
    base = orc.ar_rmsnorm(P, R, W, eps)
    for c in (0.25, 2.0, 4.0):
        Pc = [torch_bf16_bits(bits_to_f32(p) * np.float32(c)) for p in P]
        Rc = torch_bf16_bits(bits_to_f32(R) * np.float32(c))
        out, rout, s = orc.ar_rmsnorm(Pc, Rc, W, eps)
        if not np.array_equal(s, base[2] * np.float32(c)):
            fails.append(f"scale {c}: sum not scaled exactly")
        if not np.array_equal(bits_to_f32(rout), bits_to_f32(base[1]) * np.float32(c)):
            fails.append(f"scale {c}: residual_out not scaled exactly")
        d = np.abs(bits_to_f32(out).astype(np.float64) - bits_to_f32(base[0]))
        if np.any(d > BF16_REL * np.abs(bits_to_f32(base[0])) + BF16_ABS):
            fails.append(f"scale {c}: out moved by {float(d.max())}")
    return fails


def check_threads_do_not_matter(orc):
    rng = np.random.default_rng(4)
    P, R, W = random_case(rng, 3, 37, 64)
    a = orc.ar_rmsnorm(P, R, W, 1e-6, threads=1)
    b = orc.ar_rmsnorm(P, R, W, 1e-6, threads=5)
    if not all(np.array_equal(x, y) for x, y in zip(a, b)):
        return ["row-parallel oracle run differs from the serial one"]
    return []


ALL_CHECKS = [
    check_bf16_rounding_vs_torch,
    check_bf16_rounding_by_hand,
    check_hand_rows,
    check_tree_order_would_differ,
    check_brute_force_dyadic,
    check_sum_error_bound,
    check_n1_is_textbook_rmsnorm,
    check_rms_invariant,
    check_scale_invariance,
    check_threads_do_not_matter,
]


def run_all(orc):
    fails = []
    for chk in ALL_CHECKS:
        try:
            fails += [f"{chk.__name__}: {f}" for f in chk(orc)]
        except Exception as e:  # a crash is a failure too
            fails.append(f"{chk.__name__}: raised {type(e).__name__}: {e}")
    return fails
