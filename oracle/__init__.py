"""Float64 CPU oracle for the tensor-parallel MLP block and its sequence-parallel form.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package: only
the tests, the smoke check and the benchmark's CPU-baseline leg may call it. It
shares no code with the CUDA library (no kernels, headers, constants or helpers);
its only common ground with the GPU path is the seeded input generator in
``tensor_transformer_mlp_gb300.workloads``, which holds none of the arithmetic.

What it computes, and which passage of the source pages it follows:

* ``mlp``: the unsharded definition Z = X A, Y = gelu(Z), O = Y B and the four
  gradients D = (G B^T) * gelu'(Z), dA = X^T D, dB = Y^T G, dX = D A^T
  ("024 | Megatron-LM: 按矩阵结构切分 Transformer", section 二, the
  block "前向少通信，反向为何仍要一次归约？"), plus an explicitly sharded restatement
  of the same quantities (eqs. (1)(2) of the SenseParrots model-parallel note,
  section 2.1) used only to pin the shard-sum invariant.
* ``sp``: LayerNorm with torch semantics, the splitmix64 counter-hash dropout mask,
  and the sequence-parallel block (placement diagram of "Megatron-SP 机制",
  section "通信插在层内什么位置？").
* ``attention``: the tensor-parallel self-attention block (column-parallel QKV with heads split
  across shards, softmax(Q K^T / sqrt(head_dim)) V per head, row-parallel output projection) and
  its gradients, from the SenseParrots note's parallel attention code (section 2.1.1) and the
  "Attention 层" section of the "Megatron 训练" notes.
* ``collectives``: host "ranks" for all-reduce, all-gather and reduce-scatter, to pin
  AllReduce = AllGather(ReduceScatter(x)) ("Megatron-SP 机制", section
  "f/g 算子怎么定义？").

Every floating-point step runs in float64 on inputs that are already rounded to
the workload's dtype. Pins (tests/test_oracle_pins.py) tie each function to
something other than itself: finite differences, torch autograd, brute force,
closed forms, the block-matrix invariants and the ReLU counterexample. The
worked example on the pages prints shapes only, so its absolute values are
parity-unpinned; every other function here is pinned.
"""
from . import attention, collectives, mlp, sp  # noqa: F401
