"""Write exact_causal_gqa.json: a tiny attention case differentiated symbolically with sympy.

The values pin the fp64 oracle from outside: this script never imports the oracle.  It builds
the forward of the page "CANN ops-transformer FlashAttnGrad 算子详解" (discosf.com/news/4863418),
§一 (S = scale·QKᵀ, P = softmax over the visible keys, Y = PV), as a sympy expression in the
input symbols, forms L = Σ dY ⊙ Y, and differentiates it exactly.  Gradients are printed with
30 significant digits.

Case: BSND, B=1, S1=3, S2=4, N1=2, N2=1 (GQA, G=2), D=3, Dv=2, scale=1/2, causal mask read as
bottom-right aligned (key j visible to query i iff j <= i + S2 - S1).  Inputs are small
rationals so the expression is exact.

Run:  python tests/golden/make_exact_golden.py   (takes about a minute)
"""
import json
import os

import sympy as sp

S1, S2, N1, N2, D, Dv = 3, 4, 2, 1, 3, 2
SCALE = sp.Rational(1, 2)


def val(seed, n):
    # deterministic small rationals in [-1, 1] (a linear congruential walk; no randomness needed)
    out, x = [], seed
    for _ in range(n):
        x = (x * 1103515245 + 12345) % 2147483648
        out.append(sp.Rational((x >> 16) % 17 - 8, 8))
    return out


def main():
    qv, kv, vv, dyv = val(1, S1 * N1 * D), val(2, S2 * N2 * D), val(3, S2 * N2 * Dv), val(4, S1 * N1 * Dv)
    qs = sp.symbols(f"q0:{S1 * N1 * D}")
    ks = sp.symbols(f"k0:{S2 * N2 * D}")
    vs = sp.symbols(f"v0:{S2 * N2 * Dv}")

    def Q(i, n, d): return qs[(i * N1 + n) * D + d]
    def K(j, n, d): return ks[(j * N2 + n) * D + d]
    def V(j, n, d): return vs[(j * N2 + n) * Dv + d]
    def dY(i, n, d): return dyv[(i * N1 + n) * Dv + d]

    G = N1 // N2
    L = 0
    Y_expr, lse_expr = {}, {}
    for n1 in range(N1):
        n2 = n1 // G
        for i in range(S1):
            keys = [j for j in range(S2) if j <= i + S2 - S1]
            s = {j: SCALE * sum(Q(i, n1, d) * K(j, n2, d) for d in range(D)) for j in keys}
            z = sum(sp.exp(s[j]) for j in keys)
            lse_expr[(n1, i)] = sp.log(z)
            for dv in range(Dv):
                y = sum(sp.exp(s[j]) / z * V(j, n2, dv) for j in keys)
                Y_expr[(i, n1, dv)] = y
                L += dY(i, n1, dv) * y

    subs = dict(zip(qs, qv))
    subs.update(zip(ks, kv))
    subs.update(zip(vs, vv))

    def ev(e):
        return sp.N(e.subs(subs), 30)

    grads = {}
    for name, syms in (("dq", qs), ("dk", ks), ("dv", vs)):
        grads[name] = [str(ev(sp.diff(L, x))) for x in syms]
    out = {
        "citation": "page 'CANN ops-transformer FlashAttnGrad 算子详解' (discosf.com/news/4863418), "
                    "§一 forward and backward equations; causal mask read as bottom-right aligned; "
                    "GQA q-head n1 uses kv-head n1 // (N1/N2)",
        "layout": "BSND", "B": 1, "S1": S1, "S2": S2, "N1": N1, "N2": N2, "D": D, "Dv": Dv,
        "softmax_scale": 0.5, "mask_mode": 1, "win_left": -1, "win_right": -1,
        "q": [str(x) for x in qv], "k": [str(x) for x in kv], "v": [str(x) for x in vv],
        "dout": [str(x) for x in dyv],
        "attn_out": [str(ev(Y_expr[(i, n, d)])) for i in range(S1) for n in range(N1) for d in range(Dv)],
        "softmax_lse": [str(ev(lse_expr[(n, i)])) for n in range(N1) for i in range(S1)],
        **grads,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exact_causal_gqa.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, ensure_ascii=False)
    print("wrote", path)


if __name__ == "__main__":
    main()
