"""The kernels' eight-key dropout hash (DropHash8 / drop_bits8 in csrc/device_common.cuh), run
on the CPU.

drop_bits8 decides eight consecutive elements at once and takes a shortcut that is exact only
outside four rare cases (a carry out of the low word of seed ^ k + gamma, a change of that low
word's bits 30-31 within the eight keys, a threshold of 2^63 or more, and a tie between the last
product's high word and the threshold's). Random inputs on
the GPU reach those cases about once in 2^32 keys, so this test compiles the helper as host
code with nvcc and checks it, bit for bit, against the float64 oracle's splitmix64 on inputs
built to land in each case, plus random ones. Dropout rule: "Megatron-SP 机制", section on the
RNG domains (each shard draws its own mask); the hash is SplitMix64 (Steele, Lea and Flood 2014).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import sp as osp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tensor_transformer_mlp_gb300", "csrc")
M64 = (1 << 64) - 1
GAMMA_LO = 0x9E3779B97F4A7C15 & 0xFFFFFFFF

HARNESS = r"""
#include <cstdio>
#include "device_common.cuh"
// drop_bits8 with the seed's low three bits as a compile-time constant, as the dropout kernels
// instantiate it.
template <int L>
unsigned with_low3(unsigned long long base, unsigned long long threshold) {
  return tpmlp::drop_bits8<L>(base, threshold);
}
int main() {
  unsigned (*by_low3[8])(unsigned long long, unsigned long long) = {
      with_low3<0>, with_low3<1>, with_low3<2>, with_low3<3>, with_low3<4>, with_low3<5>, with_low3<6>, with_low3<7>};
  unsigned long long base, threshold;
  while (std::scanf("%llx %llx", &base, &threshold) == 2) {
    unsigned full = 0;
    for (unsigned e = 0; e < 8; ++e) full |= (tpmlp::hash_below(base ^ e, threshold) ? 1u : 0u) << e;
    std::printf("%u %u %u\n", tpmlp::drop_bits8(base, threshold), by_low3[base & 7](base, threshold), full);
  }
  return 0;
}
"""


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("drop_bits")
    src, exe = d / "harness.cu", d / "harness"
    src.write_text(HARNESS)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O2", "-I", CSRC, "-I",
           os.path.join(ROOT, "include"), str(src), "-o", str(exe)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr

    def run(cases):
        text = "".join(f"{b:x} {t:x}\n" for b, t in cases)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True).stdout.split()
        got = np.array(out, dtype=np.int64).reshape(-1, 3)
        return got[:, 0], got[:, 1], got[:, 2]

    return run


def _oracle_bits(cases):
    base = np.array([b for b, _ in cases], dtype=np.uint64)
    thr = np.array([t for _, t in cases], dtype=np.uint64)
    bits = np.zeros(len(cases), dtype=np.int64)
    for e in range(8):
        bits |= (osp.splitmix64(base ^ np.uint64(e)) < thr).astype(np.int64) << e
    return bits


def _check(harness, cases):
    fast, fast_low3, full = harness(cases)
    want = _oracle_bits(cases)
    assert np.array_equal(full, want), "hash_below disagrees with the oracle"
    for got in (fast, fast_low3):
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, [(hex(cases[i][0]), hex(cases[i][1]), got[i], want[i]) for i in bad[:5]]


def test_random_keys_and_thresholds(harness):
    rng = np.random.default_rng(20)
    bases = [int(x) for x in rng.integers(0, 1 << 63, 4000, dtype=np.uint64) * 2]
    bases += [int(x) for x in rng.integers(0, 1 << 20, 1000, dtype=np.uint64)]
    thresholds = [osp.drop_threshold(p) for p in (0.0, 0.1, 0.25, 0.3, 0.49999999, 0.5, 0.75, 0.9)]
    thresholds += [1, (1 << 63) - 1, M64]
    cases = [(b, t) for b in bases for t in thresholds]
    cases += [(b, int(t)) for b, t in zip(bases, rng.integers(0, 1 << 63, len(bases), dtype=np.uint64) * 2)]
    _check(harness, cases)


def test_carry_into_high_word(harness):
    # (base & ~7) + gamma has a low word within 7 of 2^32: some of the eight keys carry.
    rng = np.random.default_rng(21)
    cases = []
    for hi in (int(x) for x in rng.integers(0, 1 << 32, 16, dtype=np.uint64)):
        for top in range(0xFFFFFFF8, 0x100000000):
            lo = (top - GAMMA_LO) & 0xFFFFFFFF
            for low3 in range(8):
                base = (hi << 32) | (lo & ~7) | low3
                for p in (0.1, 0.3, 0.5):
                    cases.append((base, osp.drop_threshold(p)))
    assert any((((b & ~7) + 0x9E3779B97F4A7C15) & 0xFFFFFFFF) > 0xFFFFFFF8 for b, _ in cases)
    _check(harness, cases)


def test_low_word_crosses_bit_30(harness):
    # (base & ~7) + gamma has a low word whose low 30 bits lie within 7 of 2^30: some of the
    # eight keys change bits 30-31 of the low word, which the shared first xor-shift assumes fixed.
    rng = np.random.default_rng(23)
    cases = []
    for hi in (int(x) for x in rng.integers(0, 1 << 32, 8, dtype=np.uint64)):
        for top2 in range(3):
            for low30 in range(0x3FFFFFF8, 0x40000000):
                lo = ((top2 << 30) | low30) - GAMMA_LO
                for low3 in range(8):
                    base = (hi << 32) | (lo & 0xFFFFFFF8) | low3
                    for p in (0.1, 0.4):
                        cases.append((base, osp.drop_threshold(p)))
    assert any(((((b & ~7) + 0x9E3779B97F4A7C15) & 0x3FFFFFFF) > 0x3FFFFFF8) for b, _ in cases)
    _check(harness, cases)


def test_threshold_ties_high_word(harness):
    # Thresholds whose high word equals a key's hash high word; the low word decides.
    rng = np.random.default_rng(22)
    cases = []
    for b in (int(x) for x in rng.integers(0, 1 << 63, 300, dtype=np.uint64)):
        for e in range(8):
            h = osp.splitmix64_scalar(b ^ e)
            hi = h & ~0xFFFFFFFF
            for lo in (0, 1, (h & 0xFFFFFFFF), (h & 0xFFFFFFFF) + 1, 0xFFFFFFFF):
                t = hi | (lo & 0xFFFFFFFF)
                cases.append((b, t))
    assert any((t >> 32) < (1 << 31) for _, t in cases)
    _check(harness, cases)
