"""Writes gelu_tanh_points.txt: the tanh form of GeLU evaluated at a few points
in 40-digit arithmetic (mpmath), independently of the oracle.

gelu(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))

The constants sqrt(2/pi) and 0.044715 are those of the tanh approximation of
GeLU (Hendrycks & Gimpel, "Gaussian Error Linear Units (GELUs)", 2016); the
page "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核与 MoQ
量化支持" (§3.2, region 3) names GeLU in the fused FFN region, and the tanh form
is the reading taken for every workload.  Run: python make_gelu_points.py
"""
import os

import mpmath

mpmath.mp.dps = 40
POINTS = ["0.5", "1", "-1", "2", "-2", "3"]


def gelu(x):
    x = mpmath.mpf(x)
    return x / 2 * (1 + mpmath.tanh(mpmath.sqrt(2 / mpmath.pi) * (x + mpmath.mpf("0.044715") * x ** 3)))


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gelu_tanh_points.txt")
    with open(out, "w") as f:
        f.write("# GeLU, tanh form: gelu(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))),\n"
                "# evaluated in 40-digit arithmetic (mpmath), independently of the oracle, by\n"
                "# make_gelu_points.py in this folder.  Constants of the tanh approximation of\n"
                "# GeLU: Hendrycks & Gimpel, \"Gaussian Error Linear Units (GELUs)\", 2016.  The\n"
                "# page \"DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核\n"
                "# 与 MoQ 量化支持\" (§3.2, region 3) names GeLU in the fused FFN region; the tanh\n"
                "# form is the reading taken for every workload.\n"
                "# columns: x  gelu_tanh(x) (20 significant digits)\n")
        for p in POINTS:
            f.write(f"{p:>5}  {mpmath.nstr(gelu(p), 20, strip_zeros=False)}\n")
    print(open(out).read())
