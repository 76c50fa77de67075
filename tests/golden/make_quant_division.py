"""Write quant_division.json: rows where the int8 quantizer's reading of the
division decides the code.

The reading (int8 KV cache, "Character.AI: inference optimization", section
05; the pages fix no rounding): s = absmax / 127 and code = clamp(round half to
even(x / s), -127, 127), each division one IEEE fp32 operation.  Two plausible
slips give other codes on the rows written here:
  * multiplying by a rounded reciprocal, x * fl(1 / s);
  * multiplying by the rounded inverse scale, x * fl(127 / absmax);
and rows with a true tie after the division (the fp32 quotient is exactly
k + 1/2 although x / s is not) tell round-half-even from round-half-away.

Expected values are computed here from the definition with exact rational
arithmetic (fractions.Fraction), each fp32 operation rounded to nearest-even
by hand, so they depend on neither the oracle nor the CUDA library.

    python tests/golden/make_quant_division.py
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "quant_division.json")
D = 128


def f32(fr: Fraction) -> np.float32:
    """The float32 nearest to an exact rational, ties to even (normal and subnormal range)."""
    if fr == 0:
        return np.float32(0.0)
    sign = -1.0 if fr < 0 else 1.0
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 23, -149)          # spacing of float32 values at this magnitude
    scaled = a / Fraction(2) ** q
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return np.float32(sign * n * 2.0 ** q)


def fr(x) -> Fraction:
    return Fraction(float(x))


def rne(f: np.float32) -> int:
    """Round a float32 to the nearest integer, ties to even (exact on float64)."""
    v = float(f)
    lo = int(np.floor(v))
    r = v - lo
    if r > 0.5 or (r == 0.5 and lo % 2 == 1):
        lo += 1
    return lo


def code(x: np.float32, s: np.float32) -> int:
    if s == 0:
        return 0
    return max(-127, min(127, rne(f32(fr(x) / fr(s)))))


def main():
    rng = np.random.default_rng(20261203)
    rows = []
    kinds = {"reciprocal": 0, "inverse_scale": 0, "tie": 0}
    while len(rows) < 16:
        amax = np.float32(rng.uniform(0.25, 8.0))
        s = f32(fr(amax) / 127)
        inv = f32(Fraction(1) / fr(s))
        inv_scale = f32(Fraction(127) / fr(amax))
        picked = []
        for _ in range(4000):
            k = int(rng.integers(-126, 126))
            x = f32(Fraction(2 * k + 1, 2) * fr(s))
            for step in range(int(rng.integers(0, 3))):
                x = np.nextafter(x, np.float32(np.inf) if rng.integers(0, 2) else np.float32(-np.inf))
            if not (0 < abs(x) < amax):
                continue
            c = code(x, s)
            q = f32(fr(x) / fr(s))
            why = []
            if rne(f32(fr(x) * fr(inv))) != c:
                why.append("reciprocal")
            if rne(f32(fr(x) * fr(inv_scale))) != c:
                why.append("inverse_scale")
            if float(q) % 1.0 in (0.5, -0.5) and fr(x) / fr(s) != fr(q):
                why.append("tie")
            if why and all(x != p[0] for p in picked):
                picked.append((x, c, why))
            if len(picked) == 6:
                break
        if len(picked) < 6:
            continue
        sign = -1.0 if rng.integers(0, 2) else 1.0
        xs = np.zeros(D, dtype=np.float32)
        xs[0] = np.float32(sign) * amax        # the absmax element sets the scale
        pos = rng.choice(np.arange(1, D), size=len(picked), replace=False)
        for (x, _, _), p in zip(picked, pos):
            xs[p] = x
        codes = [code(x, s) for x in xs]
        assert codes[0] == int(sign) * 127
        for (_, c, why), p in zip(picked, pos):
            for w in why:
                kinds[w] += 1
        rows.append({
            "x_bits": [int(v) for v in xs.view(np.uint32)],
            "scale_bits": int(np.asarray([s], dtype=np.float32).view(np.uint32)[0]),
            "codes": codes,
            "cases": [{"index": int(p), "why": why} for (_, _, why), p in zip(picked, pos)],
        })
    doc = {
        "what": "int8 quantizer rows (128 fp32 values as IEEE bit patterns) with their scale and codes",
        "source": "'Character.AI: inference optimization', 05 Quantization and cost (int8 KV cache); the pages fix "
                  "no rounding, the reading is s = absmax/127 and code = round-half-even(x/s) in IEEE fp32, "
                  "clamped to [-127, 127]",
        "written_by": "tests/golden/make_quant_division.py (exact rationals, no oracle, no CUDA)",
        "case_counts": kinds,
        "rows": rows,
    }
    with open(OUT, "w") as f:
        json.dump(doc, f, separators=(",", ":"))
        f.write("\n")
    print(OUT, kinds)


if __name__ == "__main__":
    main()
