"""Writes quintic_map.txt: the scalar map of the Newton-Schulz quintic, exactly.

One Newton-Schulz step X <- aX + b(XX^T)X + c(XX^T)^2 X acts on each singular
value of X as f(s) = a s + b s^3 + c s^5 and leaves the singular vectors alone
(DMuon technical summary, section 2.2: the iteration on the momentum-aggregated
gradient; coefficients (3.4445, -4.7750, 2.0315), the published Muon quintic,
a reading -- the pages print none).  This script iterates f in exact rational
arithmetic (Python fractions, no floating point and nothing from oracle/) for
a few starting values and prints f^k(s) for k = 1..6 with 17 significant
digits.  Run: python tests/golden/make_quintic_map.py > tests/golden/quintic_map.txt
"""
from fractions import Fraction

A, B, C = Fraction("3.4445"), Fraction("-4.7750"), Fraction("2.0315")
STARTS = ["0.001", "0.01", "0.05", "0.1", "0.25", "0.5", "0.7", "0.9", "1", "1.1"]


def f(s):
    return A * s + B * s ** 3 + C * s ** 5


print("# s  f^1(s) .. f^6(s); quintic (3.4445, -4.7750, 2.0315), exact rational iteration, 17 digits")
for s0 in STARTS:
    s = Fraction(s0)
    vals = []
    for _ in range(6):
        s = f(s)
        vals.append(f"{float(s):.17g}" if abs(s) < 10 ** 6 else "inf")
    print(s0, " ".join(vals))
