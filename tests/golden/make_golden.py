"""Write the stored expected values under tests/golden/ from the float64 oracle only.

Run from the repository root: ``python tests/golden/make_golden.py``. The worked
example of "024 | Megatron-LM: 按矩阵结构切分 Transformer" (section 二, "给两次投影标上跨卡尺寸")
fixes only its shapes (X 3x4, A 4x8, B 8x4, two shards); its values are drawn from
seed 0 by the shared input generator and every expected value comes from ``oracle``.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import mlp  # noqa: E402
from tensor_transformer_mlp_gb300 import workloads as wl  # noqa: E402


def main():
    cfg = wl.WORKED_EXAMPLE
    inp = wl.mlp_inputs(cfg)
    f = mlp.forward(inp["X"], inp["A"], inp["B"], cfg.gelu)
    b = mlp.backward(inp["X"], inp["A"], inp["B"], inp["G"], cfg.gelu)
    path = os.path.join(HERE, "worked_example_seed0.txt")
    with open(path, "w") as fh:
        fh.write("# Two-shard worked example (shapes from '024 | Megatron-LM', section 2, "
                 "'给两次投影标上跨卡尺寸'); values: seed 0 inputs, float64 oracle, erf GeLU.\n")
        for name, arr in (("X", inp["X"]), ("A", inp["A"]), ("B", inp["B"]), ("G", inp["G"]),
                          ("O", f["O"]), ("dX", b["dX"]), ("dA", b["dA"]), ("dB", b["dB"])):
            fh.write(f"{name} {arr.shape[0]} {arr.shape[1]}\n")
            for row in np.asarray(arr, np.float64):
                fh.write(" ".join(repr(float(v)) for v in row) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
