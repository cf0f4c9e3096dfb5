"""Write adam_two_steps.json: two Adam steps on scalars in exact arithmetic.

Uses only ``fractions`` and ``decimal`` (50 significant digits); it does not
import the oracle.  Update rule (bias-corrected Adam, decoupled decay 0):
    m_t = b1 m_{t-1} + (1 - b1) G_t,   v_t = b2 v_{t-1} + (1 - b2) G_t^2
    p_t = p_{t-1} - lr * (m_t / (1 - b1^t)) / (sqrt(v_t / (1 - b2^t)) + eps)
Run:  python tests/golden/make_adam_golden.py
"""
import json
import os
from decimal import Decimal, getcontext
from fractions import Fraction as F

getcontext().prec = 50


def dsqrt(fr):
    return (Decimal(fr.numerator) / Decimal(fr.denominator)).sqrt()


def dec(fr):
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def run(p0, grads, lr, b1, b2, eps):
    p = Decimal(p0)
    m = F(0)
    v = F(0)
    out = []
    for t, g in enumerate(grads, start=1):
        g = F(g)
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        m_hat = m / (1 - b1 ** t)
        v_hat = v / (1 - b2 ** t)
        p = p - dec(lr) * dec(m_hat) / (dsqrt(v_hat) + dec(eps))
        out.append({"t": t, "m": float(dec(m)), "v": float(dec(v)), "p": float(p)})
    return out


cases = []
for p0, grads, lr in [("0", ["1", "-0.5"], "0.1"),
                      ("0.25", ["-0.003", "0.002"], "0.0001"),
                      ("-1.5", ["2e-9", "-7e-9"], "0.01")]:
    b1, b2, eps = F("0.9"), F("0.999"), F("1e-8")
    cases.append({"p0": float(p0), "grads": [float(g) for g in grads],
                  "lr": float(lr), "beta1": 0.9, "beta2": 0.999, "eps": 1e-8,
                  "steps": run(p0, grads, F(lr), b1, b2, eps)})

doc = {"source": "Adam with bias correction and eps outside the square root, weight "
                 "decay 0 (Deep Dive - Tinker, 'optim_step advances adapter state': "
                 "AdamW-equivalent, default weight decay zero). Values computed in exact "
                 "rational arithmetic with a 50-digit square root.",
       "cases": cases}
path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "adam_two_steps.json")
with open(path, "w") as fh:
    json.dump(doc, fh, indent=1)
print(path)
