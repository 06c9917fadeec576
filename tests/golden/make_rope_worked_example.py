"""Writes rope_worked_example.txt from closed forms (Python's math module only).

Worked example of one RoPE rotation, LazyAttention: Efficient Retrieval-Augmented
Generation with Deferred Positional Encoding, §3.2 "Prefilling":
    k1' = k1 cos(a) - k2 sin(a),   k2' = k1 sin(a) + k2 cos(a),
with half-dimension pairs (k[i], k[i + D/2]) and a = pos * base^(-2i/D).

D = 4, base = 10000, pos = 1: the pair (x0, x2) turns by 1 rad and the pair
(x1, x3) by 10000^(-1/2) = 0.01 rad. A second example uses pos = 3 on a D = 2
vector (a single pair, angle 3 rad).
"""
import math
import pathlib

rows = []
# example 1: D=4, theta=1e4, pos=1, x=[1,2,3,4]
x = [1.0, 2.0, 3.0, 4.0]
a0, a1 = 1.0 * 10000.0 ** (-0.0 / 4), 1.0 * 10000.0 ** (-2.0 / 4)
y = [x[0] * math.cos(a0) - x[2] * math.sin(a0),
     x[1] * math.cos(a1) - x[3] * math.sin(a1),
     x[0] * math.sin(a0) + x[2] * math.cos(a0),
     x[1] * math.sin(a1) + x[3] * math.cos(a1)]
rows.append(("4", "10000", "1", x, y))
# example 2: D=2, theta=10000, pos=3, x=[0.5,-2]
x = [0.5, -2.0]
a = 3.0
y = [x[0] * math.cos(a) - x[1] * math.sin(a), x[0] * math.sin(a) + x[1] * math.cos(a)]
rows.append(("2", "10000", "3", x, y))

out = pathlib.Path(__file__).with_name("rope_worked_example.txt")
with open(out, "w") as f:
    f.write("# RoPE worked examples (closed form; see make_rope_worked_example.py)\n")
    f.write("# source: LazyAttention paper, section 3.2 'Prefilling', rotation of a half-dimension pair\n")
    f.write("# columns: head_dim theta pos | x ... | rotated x ...\n")
    for D, th, pos, x, y in rows:
        f.write(f"{D} {th} {pos} | {' '.join(repr(v) for v in x)} | {' '.join(repr(v) for v in y)}\n")
