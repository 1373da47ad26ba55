"""Writes kda_small.txt: fp64 oracle outputs for one small fixed problem.

Calls only the oracle.  The problem: K = V = 8, two value heads sharing one
query/key head, two packed sequences of lengths 2 and 4, an initial state, and
hand-picked bf16-exact inputs (no random draws), so the file can be checked on
any machine.  Layout of the file: out [1,6,2,8] then final_state [2,2,8,8],
flattened row-major, one value per line.
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kda_inputs as KI  # noqa: E402


def golden_case() -> KI.KdaInputs:
    K = V = 8
    T, H_qk, H_v = 6, 1, 2
    i = torch.arange(T * H_qk * K, dtype=torch.float32).reshape(1, T, H_qk, K)
    q = ((i % 7) - 3.0) * 0.5
    k = ((i * 3 % 11) - 5.0) * 0.25
    j = torch.arange(T * H_v * V, dtype=torch.float32).reshape(1, T, H_v, V)
    v = ((j * 5 % 13) - 6.0) * 0.125
    graw = ((j * 7 % 9) - 4.0) * 0.5
    b = torch.tensor([[[0.5, -1.0], [2.0, 0.0], [-0.5, 1.5], [1.0, -2.0], [0.25, 0.75], [-1.5, 3.0]]])
    A_log = torch.tensor([-0.5, 0.25])
    s = torch.arange(2 * H_v * V * K, dtype=torch.float32).reshape(2, H_v, V, K)
    init = ((s * 13 % 17) - 8.0) * 0.0625
    bf = lambda x: x.to(torch.bfloat16)
    return KI.KdaInputs(q=bf(q), k=bf(k), v=bf(v), graw=bf(graw), b=bf(b), A_log=A_log,
                        scale=1.0 / np.sqrt(8.0), initial_state=init,
                        cu_seqlens=torch.tensor([0, 2, 6], dtype=torch.int32), name="golden")


def main():
    import oracle
    out, fin = oracle.fwd_inputs(golden_case())
    vals = np.concatenate([out.ravel(), fin.ravel()])
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "kda_small.txt")
    np.savetxt(path, vals, fmt="%.17e")
    print(path, vals.size)


if __name__ == "__main__":
    main()
