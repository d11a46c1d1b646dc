"""Print the constants of the double-f32 exponential in sampler.cu.

Run once by hand (``python gen_exp_tables.py``); its output is pasted into
sampler.cu.  Everything is computed in 50-digit arithmetic (sympy) from the
definitions: 2^(j/64) for j = 0..63 split into a float32 head and the float32
nearest to the remainder; ln(2)/64 split into three 11-bit heads (so that
k * head is exact in float32 for |k| < 2^13) and a float32 tail; 64/ln(2)
rounded to float32.
"""

import numpy as np
import sympy as sp

D = 50


def split(v):
    h = np.float32(float(v))
    l = np.float32(float(v - sp.Float(float(h), D)))
    return h, l


def head_bits(v, bits):
    """v rounded toward zero to `bits` significant bits (exactly representable)."""
    e = sp.floor(sp.log(abs(v), 2))
    q = sp.Integer(2) ** (e - bits + 1)
    return sp.floor(v / q) * q


def main():
    print("// 2^(j/64) = hi + lo, j = 0..63")
    for j in range(64):
        h, l = split(sp.Integer(2) ** sp.Rational(j, 64))
        print(f"  {{{float(h).hex()}f, {float(l).hex()}f}},".replace("0x", "0x"))
    L = (sp.log(2) / 64).evalf(D)
    L1 = head_bits(L, 11)
    L2 = head_bits(L - L1, 11)
    L3 = head_bits(L - L1 - L2, 11)
    L4 = np.float32(float(L - L1 - L2 - L3))
    for name, v in (("L1", L1), ("L2", L2), ("L3", L3)):
        f = np.float32(float(v))
        assert sp.Float(float(f), D) == sp.Float(v, D), name  # exact
        print(f"// {name} = {float(f).hex()}")
    print(f"// L4 = {float(L4).hex()}")
    print(f"// 64/ln2 = {float(np.float32(float((64 / sp.log(2)).evalf(D)))).hex()}")


if __name__ == "__main__":
    main()
