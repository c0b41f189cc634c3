// bf16 GEMM on the 5th-generation tensor cores (tcgen05) for every contraction of the
// tensor-parallel MLP block ("024 | Megatron-LM: 按矩阵结构切分 Transformer", section 二):
//   FC1      Z = X A            epilogue: Z and Y = gelu(Z)            (column-parallel GEMM)
//   FC2      O = Y B            K-loop over all t shards = the f-bar sum  (row-parallel GEMM)
//   dgrad-1  D = (G B^T) * gelu'(Z)
//   wgrad    dB = Y^T G, dA = X^T D                 (fp32 out, K = tokens)
//   dgrad-2  dX = D A^T         K-loop over all t shards = the f sum
//
// Two persistent kernels, one CTA per SM, sharing the epilogue code:
//   gemm_bf16_pair_kernel (plain GEMMs): 256 x 256 tiles on clusters of two SMs
//               (tcgen05 cta_group::2), 6-stage ring of 32 KB per SM, paced pairs
//   gemm_bf16_wide_kernel (plain GEMMs whose wave count favours it): 256 x 512 tiles on
//               SM pairs, 4-stage ring of 48 KB per SM, 25 % fewer operand bytes per FLOP
//   gemm_bf16_kernel (batched GEMMs, or all of them when tpmlp_set_gemm_variant asks): 128 x 256
//               tiles on one SM with a 4-stage ring of 48 KB, or 128 x 128 tiles with a
//               6-stage ring of 32 KB for the batched GEMMs whose N is at most 128
// The batched launches serve the attention block ("SenseParrots" model-parallel note, section
// 2.1.1): per (batch, head) the score GEMM Q K^T, whose epilogues compute the softmax in two
// passes (row statistics, then P), the dP GEMM, whose epilogue forms dS, and P V, P^T dO, dS K,
// dS^T Q.
// Warp roles in both:
//   warp 0      one thread issues TMA tile loads into the shared-memory ring
//   warp 1      one thread issues tcgen05.mma (K=16 steps) into a tensor-memory
//               accumulator; two accumulators (2 x 256 columns) let the epilogue of one
//               tile overlap the main loop of the next
//   warps 2..9  epilogue: tcgen05.ld the fp32 tile, apply the fused op, store through a
//               per-warp shared-memory transpose in whole 128-byte lines (two warps per
//               tensor-memory lane quarter, each taking half of the 256 columns)
// Operands are staged with 128-byte swizzle; K-major and MN-major layouts are both
// read in place through the descriptors' major-ness bits, so no operand is transposed
// in memory. Every mbarrier wait is bounded (kWaitLimitNs); on expiry the kernel
// records a timeout, drains its own copies and MMAs, frees tensor memory and returns.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "device_common.cuh"

namespace tpmlp {
namespace {

// GEMM variant for the plain (non-batched) GEMMs, process-wide; set only through
// tpmlp_set_gemm_variant (comparison and testing). Defaults: SM-pair kernel, paced, default band.
std::atomic<int> g_pair_kernel{1};
std::atomic<int> g_pair_pacing{1};
std::atomic<int> g_pair_group{0};

constexpr int BM = 128;
constexpr int BN = 256;  // tile width of the pair kernel and the one-SM kernel's wide variant
constexpr int BK = 64;   // one 128-byte swizzle span of bf16
constexpr int UMMA_K = 16;
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KiB
constexpr int MN_BOX_BYTES = 64 * BK * 2;  // one 64(MN) x 64(K) box of an MN-major operand
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = NUM_ACC * BN;  // 512: all of tensor memory (pair kernel)
constexpr int NUM_EPI_WARPS = 8;  // two warps per tensor-memory lane quarter, each half the columns
constexpr int NUM_EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int NUM_THREADS = 64 + NUM_EPI_THREADS;
constexpr int GROUP_M = 16;
constexpr int BARRIER_BYTES = 256;
// Per epilogue warp: 32 rows x 128 bytes, used to turn the one-row-per-thread layout of
// tcgen05.ld into line-wide global stores (kEpiStore, kEpiStoreF32).
constexpr int EPI_STAGE_BYTES = 32 * 128;

// One-SM kernel configurations by tile width: 128 x 256 tiles with a 4-stage ring, or 128 x 128
// tiles (for N <= 128, e.g. N = head_dim) with a 6-stage ring and half the tensor memory.
constexpr int AUX_BUF_BYTES = 32 * 128;  // one 32-row x 64-column bf16 block
// kAuxBufs > 0 (the batched softmax and dS epilogues): each epilogue warp owns that many 4 KB
// buffers for TMA loads of P and TMA stores of its output instead of the generic staging buffer,
// and the ring shrinks to 4 stages with 1 buffer a warp, 3 with 2, 2 with 4 (the score-shaped
// GEMMs have K = head_dim = two k-blocks, so with 2 stages the next tile's operands cannot be
// loaded before the current tile's MMAs have freed a stage: the softmax pass measured 128.7 us
// with 2 stages and 4 buffers, 115.3 us with 3 stages and 2; with its later epilogue changes
// 103.6 us with 3 stages and 2 buffers, 101.3 us with 4 stages and 1).
template <int BN_T, int kAuxBufs = 0>
struct OneSm {
  static constexpr bool kAux = kAuxBufs > 0;
  static constexpr int kBN = BN_T;
  static constexpr int kStages = kAux ? (kAuxBufs >= 4 ? 2 : (kAuxBufs >= 2 ? 3 : 4)) : (BN_T == 256 ? 4 : 6);
  static constexpr int kStageBytes = A_STAGE_BYTES + BN_T * BK * 2;
  static constexpr int kEpiStageBytes = kAux ? 0 : NUM_EPI_WARPS * EPI_STAGE_BYTES;
  static constexpr int kAuxBytes = NUM_EPI_WARPS * kAuxBufs * AUX_BUF_BYTES;
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiStageBytes + kAuxBytes + BARRIER_BYTES +
                                    1024;  // + alignment slack
  static constexpr int kTmemCols = NUM_ACC * BN_T;  // a power of two, >= 32
  static constexpr int kEpiChunks = BN_T / 32 / (NUM_EPI_WARPS / 4);
  static_assert(BN_T == 256 || BN_T == 128, "tile widths");
  static_assert(kStageBytes % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert((2 * kStages + 2 * NUM_ACC + 1 + (kAux ? 2 * NUM_EPI_WARPS : 0)) * 8 + 4 <= BARRIER_BYTES,
                "barrier area");
};

struct TileSched {
  int num_mb, num_nb, num_tiles;
  __device__ __forceinline__ void coords(int tile, int& mb, int& nb) const {
    const int group_size = GROUP_M * num_nb;
    const int group = tile / group_size;
    const int first_mb = group * GROUP_M;
    const int gsz = min(num_mb - first_mb, GROUP_M);
    const int in_group = tile - group * group_size;
    mb = first_mb + in_group % gsz;
    nb = in_group / gsz;
  }
};

__device__ __forceinline__ int64_t remap_row(const RowRemap& rm, int64_t r) {
  if (!rm.enabled) return r;
  const int64_t bi = r / rm.s;
  const int64_t si = r - bi * rm.s;
  const int64_t j = si / rm.s_per_shard;
  const int64_t l = si - j * rm.s_per_shard;
  return (j * rm.b + bi) * rm.s_per_shard + l;
}

// Device form of a batched launch: batch sizes, the tensor-map coordinate slot (1..3) that
// takes each operand's row index and batch indices, the output offsets per batch index and
// the accumulator scale.
struct BatchDev {
  int nz1, nz2;
  int a_row, a_z1, a_z2;
  int b_row, b_z1, b_z2;
  int x_row, x_z1, x_z2;  // slots of the aux (P) tensor map, kEpiSoftmaxGrad
  int64_t out_z1, out_z2;
  float alpha;
};

// GeLU and GeLU' epilogue steps for the GeLU kinds other than the tanh form (eight accumulator
// values as raw bits; for GeLU', z holds the eight bf16 inputs and the result is acc * gelu'(z)),
// packed to bf16. Kept out of line: inlined and unrolled, the erf form's registers would add to
// the tanh path's in the same kernel.
__device__ __noinline__ uint4 gelu_other8(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4, uint32_t a5,
                                          uint32_t a6, uint32_t a7, int kind) {
  const uint32_t a[8] = {a0, a1, a2, a3, a4, a5, a6, a7};
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = pack_bf16x2(gelu_f<false>(__uint_as_float(a[2 * i]), kind), gelu_f<false>(__uint_as_float(a[2 * i + 1]), kind));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __noinline__ uint4 dgelu_other8(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4, uint32_t a5,
                                           uint32_t a6, uint32_t a7, uint4 z, int kind) {
  const uint32_t a[8] = {a0, a1, a2, a3, a4, a5, a6, a7};
  const uint32_t zw[4] = {z.x, z.y, z.z, z.w};
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 zf = unpack_bf16x2(zw[i]);
    w[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * gelu_grad_f<false>(zf.x, kind),
                       __uint_as_float(a[2 * i + 1]) * gelu_grad_f<false>(zf.y, kind));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Applies the epilogues that read as well as write (kEpiAccumF32, kEpiDropoutResidual) to
// 32 consecutive accumulator columns of one row.
template <int EPI>
__device__ __forceinline__ void epilogue_row32(const EpiParams& ep, int64_t row, int col0, int N,
                                               const uint32_t (&v)[32]) {
  static_assert(EPI == kEpiAccumF32 || EPI == kEpiDropoutResidual, "the other kinds are staged");
  uint32_t drop_bits = 0;  // kEpiDropoutResidual: one mask word per 32 columns
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int col = col0 + g * 8;
    if (col >= N) break;
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __uint_as_float(v[g * 8 + i]);
    if constexpr (EPI == kEpiAccumF32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(ep.out) + row * ep.ldo + col);
      const float4 o0 = dst[0], o1 = dst[1];
      dst[0] = make_float4(o0.x + a[0], o0.y + a[1], o0.z + a[2], o0.w + a[3]);
      dst[1] = make_float4(o1.x + a[4], o1.y + a[5], o1.z + a[6], o1.w + a[7]);
    } else if constexpr (EPI == kEpiDropoutResidual) {
      const int64_t prow = remap_row(ep.remap, row);
      const int64_t off = prow * ep.ldo + col;
      const uint4 xr = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ep.aux) + off);
      const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
      // k0 = row * ldo + col is a multiple of 8, so the eight keys are (seed ^ k0) ^ e
      const uint32_t bits = drop_bits8(ep.drop.seed ^ static_cast<uint64_t>(row * ep.ldo + col), ep.drop.threshold);
      drop_bits |= bits << (g * 8);
      float o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 xf = unpack_bf16x2(xw[i]);
        o[2 * i] = (bits >> (2 * i)) & 1u ? xf.x : fmaf(a[2 * i], ep.drop.scale, xf.x);
        o[2 * i + 1] = (bits >> (2 * i + 1)) & 1u ? xf.y : fmaf(a[2 * i + 1], ep.drop.scale, xf.y);
      }
      uint4 pk = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                            pack_bf16x2(o[6], o[7]));
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ep.out) + off) = pk;
    }
  }
  if constexpr (EPI == kEpiDropoutResidual) {
    // N is a multiple of 32 here, so the 32 columns are whole and form one aligned mask word.
    if (ep.drop.mask_bits) ep.drop.mask_bits[static_cast<uint64_t>(row * ep.ldo + col0) >> 5] = drop_bits;
  }
}

// Store path of the staged epilogues (bf16: 64 columns, fp32: 32 columns per call): each thread
// holds 128 bytes of its own row in seg[]; they go through the warp's shared-memory buffer
// (16-byte segments XOR-swizzled by row, so both phases are free of bank conflicts) and leave
// as 8 rows x 128 contiguous bytes per store instruction instead of 32 rows x 16 bytes.
// prow is this lane's destination row (-1 past M); every lane of the warp must call this.
template <bool F32OUT>
__device__ __forceinline__ void store_staged(uint8_t* buf, const uint4 (&seg)[8], int lane, int64_t prow, void* out,
                                             int64_t ldo, int col0, int N) {
#pragma unroll
  for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = seg[j];
  __syncwarp();
  constexpr int kElemsPerSeg = F32OUT ? 4 : 8;
  const int j = lane & 7;
  const int col = col0 + j * kElemsPerSeg;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const uint4 val = *reinterpret_cast<const uint4*>(buf + r * 128 + ((j ^ (r & 7)) << 4));
    const int64_t pr = __shfl_sync(0xffffffffu, prow, r);
    if (pr >= 0 && col < N) {
      if constexpr (F32OUT) {
        *reinterpret_cast<uint4*>(static_cast<float*>(out) + pr * ldo + col) = val;
      } else {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + pr * ldo + col) = val;
      }
    }
  }
  __syncwarp();
}

// The bulk-copy form of store_staged, for outputs with a tensor map (rows not remapped): the
// warp's 32 rows x 128 bytes go into its staging buffer in the 128-byte-swizzled layout of the
// map's 32-row box, and lane 0 stores the block with one tensor copy (parts past M or N are not
// written), so the warp moves on without waiting for the global writes. The buffer is rewritten
// only once the previous copy out of it has read it (buf_acquire).
__device__ __forceinline__ void buf_acquire(int lane) {
  if (lane == 0) bulk_wait_group_read<0>();
  __syncwarp();
}

__device__ __forceinline__ void store_tma(uint8_t* buf, const uint4 (&seg)[8], int lane, const CUtensorMap* map,
                                          int col0, int row0) {
  buf_acquire(lane);
#pragma unroll
  for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = seg[j];
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, col0, row0);
    bulk_commit_group();
  }
}

// The inverse of store_staged for bf16 (load_staged_bf16), in two steps. issue_block_loads: the
// warp reads 32 rows x 64 columns of src with line-wide loads (8 rows x 128 bytes per
// instruction; lane gets rows i*4 + lane/8, segment lane%8; zeros past M or N).
// transpose_block: through the warp's staging buffer, each thread receives its own row's 128
// bytes in seg[].
__device__ __forceinline__ void issue_block_loads(uint4 (&r8)[8], int lane, int64_t prow, const void* src, int64_t ldo,
                                                  int col0, int N) {
  const int col = col0 + (lane & 7) * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const int64_t pr = __shfl_sync(0xffffffffu, prow, r);
    r8[i] = make_uint4(0, 0, 0, 0);
    if (pr >= 0 && col < N) r8[i] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + pr * ldo + col);
  }
}

__device__ __forceinline__ void transpose_block(uint8_t* buf, const uint4 (&r8)[8], uint4 (&seg)[8], int lane) {
  const int j = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    *reinterpret_cast<uint4*>(buf + r * 128 + ((j ^ (r & 7)) << 4)) = r8[i];
  }
  __syncwarp();
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) seg[jj] = *reinterpret_cast<const uint4*>(buf + lane * 128 + ((jj ^ (lane & 7)) << 4));
  __syncwarp();
}

__device__ __forceinline__ void load_staged_bf16(uint8_t* buf, uint4 (&seg)[8], int lane, int64_t prow,
                                                 const void* src, int64_t ldo, int col0, int N) {
  uint4 r8[8];
  issue_block_loads(r8, lane, prow, src, ldo, col0, N);
  transpose_block(buf, r8, seg, lane);
}

// Scale (batched) and bias (bf16 per column) for the store kinds, 8 columns at a time.
template <int EPI, bool BATCHED>
__device__ __forceinline__ void store_prologue8(const EpiParams& ep, int col, bool col_ok, float (&a)[8],
                                                float alpha) {
  if constexpr (BATCHED) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] *= alpha;
  }
  if constexpr (EPI == kEpiStore) {
    if (ep.bias && col_ok) {
      const uint4 bv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ep.bias) + col);
      const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 bf = unpack_bf16x2(bw[i]);
        a[2 * i] += bf.x;
        a[2 * i + 1] += bf.y;
      }
    }
  }
}

// The epilogue of one accumulator tile for one epilogue warp: its 32 tensor-memory lanes
// (rows row - lane .. row - lane + 31 of the output) and its kChunks 32-column chunks from
// c_begin, starting at output column col_tile0. buf is the warp's staging buffer; srow numbers
// the row across the batch (row statistics), nb / num_nb give the tile's N-block.
constexpr int kEpiChunks = BN / 32 / (NUM_EPI_WARPS / 4);  // 32-column chunks per warp, 256-wide tiles

// tm_out / tm_out2 (non-null: the plain store kinds in the pair kernels, rows not remapped) send
// ep.out / ep.out2 through bulk tensor stores instead of store_staged. kTmaOnly (GeLU in the pair
// kernels: both outputs always have tensor maps) compiles the bulk-store path alone. The wide
// kernel has its own GeLU' epilogue; the 256 x 256 kernel's, which overlaps the next tile's main
// loop, measured 15 % slower with bulk stores or with an L2 prefetch of Z, so it keeps both out.
template <int EPI>
constexpr bool kTmaEpi = EPI == kEpiGelu;

template <int EPI, bool BATCHED, int kChunks = kEpiChunks, bool kTmaOnly = false>
__device__ __forceinline__ void epilogue_tile(const EpiParams& ep, uint8_t* buf, int lane, int64_t row, int M, int N,
                                              int col_tile0, int c_begin, uint32_t t_row, int64_t out_off,
                                              float alpha, int64_t srow, int nb, int num_nb,
                                              const CUtensorMap* tm_out = nullptr,
                                              const CUtensorMap* tm_out2 = nullptr) {
  const int row0 = static_cast<int>(row - lane);  // the warp's first row (bulk stores)
  if constexpr (EPI == kEpiStore || EPI == kEpiStoreF32) {
    constexpr bool kF32 = EPI == kEpiStoreF32;
    constexpr int kCols = kF32 ? 32 : 64;  // 128 bytes of output per row per pass
    const int64_t prow = row < M ? remap_row(ep.remap, row) : -1;
    void* out = kF32 ? static_cast<void*>(static_cast<float*>(ep.out) + out_off)
                     : static_cast<void*>(static_cast<__nv_bfloat16*>(ep.out) + out_off);
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; c += kCols / 32) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[kCols];
      if constexpr (!kF32)
        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_wait();
      uint4 seg[8];
#pragma unroll
      for (int g = 0; g < kCols / 8; ++g) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = __uint_as_float(v[g * 8 + i]);
        store_prologue8<EPI, BATCHED>(ep, col0 + g * 8, col0 + g * 8 < N, a, alpha);
        if constexpr (kF32) {
          seg[2 * g] = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                  __float_as_uint(a[3]));
          seg[2 * g + 1] = make_uint4(__float_as_uint(a[4]), __float_as_uint(a[5]), __float_as_uint(a[6]),
                                      __float_as_uint(a[7]));
        } else {
          seg[g] = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                              pack_bf16x2(a[6], a[7]));
        }
      }
      if (tm_out)
        store_tma(buf, seg, lane, tm_out, col0, row0);
      else
        store_staged<kF32>(buf, seg, lane, prow, out, ep.ldo, col0, N);
    }
  } else if constexpr (EPI == kEpiStoreRowDot) {
    // bf16 stores as kEpiStore (64 columns per pass, staged), and each row's dot product of the
    // stored values with aux over the warp's 128 columns (one head of 128), accumulated over the
    // passes in column order; aux arrives through the staging buffer like Z in kEpiDGelu.
    const int64_t prow = row < M ? row : -1;
    float dot = 0.f;
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; c += 2) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[64];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      uint4 os[8];
      load_staged_bf16(buf, os, lane, prow, ep.aux, ep.ldo, col0, N);
      tmem_ld_wait();
      uint4 seg[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint32_t ow[4] = {os[g].x, os[g].y, os[g].z, os[g].w};
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w[i] = pack_bf16x2(__uint_as_float(v[g * 8 + 2 * i]), __uint_as_float(v[g * 8 + 2 * i + 1]));
          const float2 d2 = unpack_bf16x2(w[i]), o2 = unpack_bf16x2(ow[i]);
          dot = fmaf(d2.x, o2.x, dot);
          dot = fmaf(d2.y, o2.y, dot);
        }
        seg[g] = make_uint4(w[0], w[1], w[2], w[3]);
      }
      store_staged<false>(buf, seg, lane, prow, ep.out, ep.ldo, col0, N);
    }
    if (row < M) {
      const int64_t bi = row / ep.rowdot_s, si = row - bi * ep.rowdot_s;
      const int j = (col_tile0 + c_begin * 32) / 128;
      ep.rowdot[(bi * ep.rowdot_heads + j) * ep.rowdot_s + si] = dot;
    }
  } else if constexpr (EPI == kEpiGelu) {
    // Z (optional) and Y = gelu(Z), 64 columns per pass, both through the staging buffer.
    const int64_t prow = row < M ? row : -1;
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; c += 2) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[64];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      // Z first (bias added in place in v), so its store is under way while Y is computed.
      uint4 zs[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = __uint_as_float(v[g * 8 + i]);
        store_prologue8<kEpiStore, false>(ep, col0 + g * 8, col0 + g * 8 < N, a, 1.f);  // bias1
#pragma unroll
        for (int i = 0; i < 8; ++i) v[g * 8 + i] = __float_as_uint(a[i]);
        zs[g] = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                           pack_bf16x2(a[6], a[7]));
      }
      if (ep.out) {
        if constexpr (kTmaOnly)
          store_tma(buf, zs, lane, tm_out, col0, row0);
        else
          store_staged<false>(buf, zs, lane, prow, ep.out, ep.ldo, col0, N);
      }
      uint4 ys[8];
      if (ep.gelu == kGeluTanh) {  // uniform: pairs of elements on the f32x2 path
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint32_t yw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 y2 = f2_split(gelu_tanh2(f2_make(__uint_as_float(v[g * 8 + 2 * i]),
                                                          __uint_as_float(v[g * 8 + 2 * i + 1]))));
            yw[i] = pack_bf16x2(y2.x, y2.y);
          }
          ys[g] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
        }
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g)
          ys[g] = gelu_other8(v[g * 8], v[g * 8 + 1], v[g * 8 + 2], v[g * 8 + 3], v[g * 8 + 4], v[g * 8 + 5],
                              v[g * 8 + 6], v[g * 8 + 7], ep.gelu);
      }
      if constexpr (kTmaOnly)
        store_tma(buf, ys, lane, tm_out2, col0, row0);
      else
        store_staged<false>(buf, ys, lane, prow, ep.out2, ep.ldo, col0, N);
    }
  } else if constexpr (EPI == kEpiRowStats) {
    // Online max / sum of exp over the warp's 128 columns of the row, in base 2: with
    // c = alpha * log2(e) > 0, y = acc * c, the running (m, l) are max y and sum 2^(y - m); per
    // 32-column chunk the sum is rescaled to the new maximum. max(acc) * c = max(acc * c) since
    // c > 0, so the max is taken on the raw accumulators; 2^(y - m) is ex2(fma(acc, c, -m)).
    // Columns past N do not count (only a ragged last chunk checks them).
    const float c2 = alpha * kLog2e;
    float m = -INFINITY, l = 0.f;
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; ++c) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[32];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), v);
      tmem_ld_wait();
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
      if (col0 + 32 > N) {  // uniform across the warp
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i >= N) x[i] = -INFINITY;
      }
      float c4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int i = 4; i < 32; ++i) c4[i & 3] = fmaxf(c4[i & 3], x[i]);
      const float mn = fmaxf(m, fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3])) * c2);
      // y - mn = fma(acc, c, -mn) and the sums on fp32 pairs (f32x2): two accumulator pairs
      const F2 c22 = f2_make(c2, c2), nmn = f2_make(-mn, -mn);
      F2 s2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 t = f2_split(f2_fma(f2_make(x[2 * i], x[2 * i + 1]), c22, nmn));
        s2[i & 1] = f2_add(s2[i & 1], f2_make(ex2_approx(t.x), ex2_approx(t.y)));
      }
      const float2 a = f2_split(s2[0]), b = f2_split(s2[1]);
      l = l * ex2_approx(m - mn) + ((a.x + b.x) + (a.y + b.y));
      m = mn;
    }
    if (row < M) {
      const int half = c_begin / kChunks;
      static_cast<float2*>(ep.stats)[srow * (2 * num_nb) + 2 * nb + half] = make_float2(m, l);
    }
  } else if constexpr (EPI == kEpiSoftmax) {
    // P = 2^(acc * c - M) / L = 2^(acc * c - (M + log2 L)) with the row's combined base-2
    // statistics (rowvec .x = M + log2 L), 64 columns per pass, staged.
    const float c2 = alpha * kLog2e;
    const float2 st = row < M ? static_cast<const float2*>(ep.rowvec)[srow] : make_float2(0.f, 0.f);
    const int64_t prow = row < M ? row : -1;
    void* out = static_cast<__nv_bfloat16*>(ep.out) + out_off;
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; c += 2) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[64];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      uint4 seg[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = ex2_approx(fmaf(__uint_as_float(v[g * 8 + i]), c2, -st.x));
        seg[g] = make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                            pack_bf16x2(p[6], p[7]));
      }
      store_staged<false>(buf, seg, lane, prow, out, ep.ldo, col0, N);
    }
  } else if constexpr (EPI == kEpiSoftmaxGrad) {
    // dS = escale * P * (dP - D): P read and dS written 64 columns at a time through the staging buffer.
    // escale * (acc * alpha - D) = acc * a2 - d2: one FFMA and one FMUL per element.
    const float a2 = alpha * ep.escale;
    const float d2 = (row < M ? static_cast<const float*>(ep.rowvec)[srow] : 0.f) * ep.escale;
    const int64_t prow = row < M ? row : -1;
    const void* pin = static_cast<const __nv_bfloat16*>(ep.aux) + out_off;
    void* out = static_cast<__nv_bfloat16*>(ep.out) + out_off;
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; c += 2) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[64];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      uint4 ps[8];
      load_staged_bf16(buf, ps, lane, prow, pin, ep.ldo, col0, N);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 8; ++g) {  // dS overwrites P in place
        uint32_t* w = reinterpret_cast<uint32_t*>(&ps[g]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 pf = unpack_bf16x2(w[i]);
          w[i] = pack_bf16x2(pf.x * fmaf(__uint_as_float(v[g * 8 + 2 * i]), a2, -d2),
                             pf.y * fmaf(__uint_as_float(v[g * 8 + 2 * i + 1]), a2, -d2));
        }
      }
      store_staged<false>(buf, ps, lane, prow, out, ep.ldo, col0, N);
    }
  } else if constexpr (EPI == kEpiDGelu) {
    // D = acc * gelu'(Z): Z read and D written 64 columns at a time through the staging buffer.
    const int64_t prow = row < M ? row : -1;
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; c += 2) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[64];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32), *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      uint4 zs[8];
      load_staged_bf16(buf, zs, lane, prow, ep.aux, ep.ldo, col0, N);
      tmem_ld_wait();
      if (ep.gelu == kGeluTanh) {  // uniform: pairs of elements on the f32x2 path; D overwrites Z in place
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint32_t* w = reinterpret_cast<uint32_t*>(&zs[g]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const F2 z2 = f2_make(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
            const float2 d2 = f2_split(f2_mul(f2_make(__uint_as_float(v[g * 8 + 2 * i]),
                                                      __uint_as_float(v[g * 8 + 2 * i + 1])),
                                              gelu_grad_tanh2(z2)));
            w[i] = pack_bf16x2(d2.x, d2.y);
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g)
          zs[g] = dgelu_other8(v[g * 8], v[g * 8 + 1], v[g * 8 + 2], v[g * 8 + 3], v[g * 8 + 4], v[g * 8 + 5],
                               v[g * 8 + 6], v[g * 8 + 7], zs[g], ep.gelu);
      }
      store_staged<false>(buf, zs, lane, prow, ep.out, ep.ldo, col0, N);
    }
  } else {
#pragma unroll 1
    for (int c = c_begin; c < c_begin + kChunks; ++c) {
      const int col0 = col_tile0 + c * 32;
      if (col0 >= N) break;  // uniform across the warp
      uint32_t v[32];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), v);
      tmem_ld_wait();
      if (row < M) epilogue_row32<EPI>(ep, row, col0, N, v);
    }
  }
}

// Per-warp TMA buffers of the batched epilogues: kEpiSoftmax stores P through one (its ring gets
// the room for a fourth stage); kEpiSoftmaxGrad loads P through two and stores dS through two more.
constexpr int kSoftmaxStoreBufs = 1;
template <int EPI, bool BATCHED>
__host__ __device__ constexpr int aux_bufs() {
  return !BATCHED ? 0 : (EPI == kEpiSoftmax ? kSoftmaxStoreBufs : (EPI == kEpiSoftmaxGrad ? 4 : 0));
}

// One TMA tile load: 2-D map for plain launches; 4-D map (inner, then row and batch indices in
// the slots recorded in BatchDev) for batched ones.
template <bool BATCHED>
__device__ __forceinline__ void load_tile(void* dst, const CUtensorMap* map, uint64_t* bar, int inner, int row, int z1,
                                          int z2, int s_row, int s_z1, int s_z2) {
  if constexpr (!BATCHED) {
    tma_load_2d(dst, map, bar, inner, row);
  } else {
    const int c1 = s_row == 1 ? row : (s_z1 == 1 ? z1 : z2);
    const int c2 = s_row == 2 ? row : (s_z1 == 2 ? z1 : z2);
    const int c3 = s_row == 3 ? row : (s_z1 == 3 ? z1 : z2);
    (void)s_z2;
    tma_load_4d(dst, map, bar, inner, c1, c2, c3);
  }
}

template <bool A_MN, bool B_MN, int EPI, bool BATCHED = false, int BN_T = 256>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_aux, const __grid_constant__ CUtensorMap tmap_out,
                     int M, int N, int K, EpiParams ep, unsigned int* status, BatchDev bd) {
  // The batched softmax and dS epilogues move P and dS by TMA through per-warp buffers
  // (tmap_aux: P to load, tmap_out: the output to store).
  constexpr int kAuxBufs = aux_bufs<EPI, BATCHED>();
  constexpr bool kAux = kAuxBufs > 0;
  using Cfg = OneSm<BN_T, kAuxBufs>;
  constexpr int BN = Cfg::kBN, STAGES = Cfg::kStages, STAGE_BYTES = Cfg::kStageBytes, TMEM_COLS = Cfg::kTmemCols;
  constexpr int kChunks = Cfg::kEpiChunks;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* epi_stage = smem + STAGES * STAGE_BYTES;
  uint8_t* aux_buf = epi_stage + Cfg::kEpiStageBytes;  // 1024-byte aligned (128-byte swizzle)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(aux_buf + Cfg::kAuxBytes);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;
  uint64_t* tempty_bar = tfull_bar + NUM_ACC;
  uint64_t* drain_bar = tempty_bar + NUM_ACC;
  uint64_t* aux_bar = drain_bar + 1;  // kAux: two per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_bar + (kAux ? 2 * NUM_EPI_WARPS : 0));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  TileSched sched;
  sched.num_mb = (M + BM - 1) / BM;
  sched.num_nb = (N + BN - 1) / BN;
  sched.num_tiles = sched.num_mb * sched.num_nb;
  const int tiles_per_batch = sched.num_tiles;
  const int total_tiles = BATCHED ? tiles_per_batch * bd.nz1 * bd.nz2 : tiles_per_batch;
  // tile -> (batch index, M block, N block); batch-major so neighbouring tiles share a batch
  auto tile_coords = [&](int tile, int& z1, int& z2, int& mb, int& nb) {
    int z = 0;
    if constexpr (BATCHED) {
      z = tile / tiles_per_batch;
      tile -= z * tiles_per_batch;
    }
    z1 = BATCHED ? z % bd.nz1 : 0;
    z2 = BATCHED ? z / bd.nz1 : 0;
    sched.coords(tile, mb, nb);
  };
  const int num_kb = (K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
#pragma unroll
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], NUM_EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    if constexpr (kAux)
      for (int i = 0; i < 2 * NUM_EPI_WARPS; ++i) mbar_init(&aux_bar[i], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    if constexpr (kAux) {
      tma_prefetch_desc(&tmap_aux);
      tma_prefetch_desc(&tmap_out);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int kiter = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        int z1, z2, mb, nb;
        tile_coords(tile, z1, z2, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb) {
          const int s = kiter % STAGES;
          const uint32_t parity = ((kiter / STAGES) & 1) ^ 1;
          if (!mbar_wait(&empty_bar[s], parity, status, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], STAGE_BYTES);
          uint8_t* sa = smem + s * STAGE_BYTES;
          uint8_t* sb = sa + A_STAGE_BYTES;
          if constexpr (!A_MN) {
            load_tile<BATCHED>(sa, &tmap_a, &full_bar[s], kb * BK, mb * BM, z1, z2, bd.a_row, bd.a_z1, bd.a_z2);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              load_tile<BATCHED>(sa + j * MN_BOX_BYTES, &tmap_a, &full_bar[s], mb * BM + j * 64, kb * BK, z1, z2,
                                 bd.a_row, bd.a_z1, bd.a_z2);
          }
          if constexpr (!B_MN) {
            load_tile<BATCHED>(sb, &tmap_b, &full_bar[s], kb * BK, nb * BN, z1, z2, bd.b_row, bd.b_z1, bd.b_z2);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              load_tile<BATCHED>(sb + j * MN_BOX_BYTES, &tmap_b, &full_bar[s], nb * BN + j * 64, kb * BK, z1, z2,
                                 bd.b_row, bd.b_z1, bd.b_z2);
          }
          ++kiter;
        }
      }
      if (!ok) {
        // Wait (bounded) for the copies still in flight before shared memory goes away.
        for (int k = max(0, kiter - STAGES); k < kiter; ++k)
          mbar_wait(&full_bar[k % STAGES], (k / STAGES) & 1, status, 2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      int kiter = 0, it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(&tempty_bar[acc], (use & 1) ^ 1, status, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          const int s = kiter % STAGES;
          if (!mbar_wait(&full_bar[s], (kiter / STAGES) & 1, status, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t b_base = a_base + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // K-major: a K16 step is 32 bytes along the 128-byte row; 8-row groups 1024 B apart.
            // MN-major: a K16 step is 16 rows of 128 bytes; 64-wide MN blocks one box apart.
            const uint64_t adesc = A_MN ? smem_desc_sw128(a_base + kk * 2048, MN_BOX_BYTES, 1024)
                                        : smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(b_base + kk * 2048, MN_BOX_BYTES, 1024)
                                        : smem_desc_sw128(b_base + kk * 32, 16, 1024);
            umma_bf16(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty_bar[s]);  // frees the stage once these MMAs have read it
          ++kiter;
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);  // accumulator ready for the epilogue
      }
      // Every MMA this thread issued must finish before tensor memory is freed.
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, status, 5);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // the tensor-memory lane quarter this warp may access
    const int c_begin = ((warp - 2) / 4) * kChunks;
    // Coordinates of a batched tensor map for (inner, row, z1, z2), slots as recorded in bd.
  auto aux_coords = [&](int inner, int row, int z1, int z2, int (&cc)[4]) {  // selects, no local memory
    cc[0] = inner;
    cc[1] = bd.x_row == 1 ? row : (bd.x_z1 == 1 ? z1 : z2);
    cc[2] = bd.x_row == 2 ? row : (bd.x_z1 == 2 ? z1 : z2);
    cc[3] = bd.x_row == 3 ? row : (bd.x_z1 == 3 ? z1 : z2);
  };
  if constexpr (kAux && EPI == kEpiSoftmax) {
      // P = 2^(acc * c - M) / L = 2^(acc * c - (M + log2 L)), one FFMA and one ex2 per score
      // (the row statistics carry M + log2 L), written by TMA stores: each 64-column pass of the warp's 32 rows
      // goes into one of its kSoftmaxStoreBufs 4 KB buffers in the 128-byte-swizzled layout the
      // store expects, and lane 0 issues the store; a buffer is reused once the store
      // kSoftmaxStoreBufs passes back has read it. The row statistics of the next tile are
      // loaded while this one is processed, and the warp's four 32-column tensor-memory loads
      // are double-buffered (chunk j + 1 in flight while chunk j is converted).
      uint8_t* sb = aux_buf + (warp - 2) * kAuxBufs * AUX_BUF_BYTES;
      const float c2 = bd.alpha * kLog2e;
      auto load_stats = [&](int tile) {
        int z1, z2, mb, nb;
        tile_coords(tile, z1, z2, mb, nb);
        const int64_t row = static_cast<int64_t>(mb) * BM + q * 32 + lane;
        const int64_t srow = (static_cast<int64_t>(z2) * bd.nz1 + z1) * M + row;
        return row < M ? static_cast<const float2*>(ep.rowvec)[srow] : make_float2(0.f, 0.f);
      };
      int nstore = 0;
      int it = 0;
      float2 st_next = blockIdx.x < total_tiles ? load_stats(blockIdx.x) : make_float2(0.f, 0.f);
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
        const float2 st = st_next;
        if (tile + static_cast<int>(gridDim.x) < total_tiles) st_next = load_stats(tile + gridDim.x);
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        const bool ok = mbar_wait(&tfull_bar[acc], use & 1, status, 6);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        int z1, z2, mb, nb;
        tile_coords(tile, z1, z2, mb, nb);
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
        uint32_t va[32], vb[32];
        uint4 seg[8];
        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c_begin * 32), va);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tmem_ld_wait();
          uint32_t(&cur)[32] = (j & 1) ? vb : va;
          uint32_t(&nxt)[32] = (j & 1) ? va : vb;
          if (j < 3) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>((c_begin + j + 1) * 32), nxt);
          const F2 c22 = f2_make(c2, c2), nst = f2_make(-st.x, -st.x);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // the exponent arguments on fp32 pairs
              const float2 t = f2_split(f2_fma(f2_make(__uint_as_float(cur[g * 8 + 2 * i]),
                                                       __uint_as_float(cur[g * 8 + 2 * i + 1])),
                                               c22, nst));
              w[i] = pack_bf16x2(ex2_approx(t.x), ex2_approx(t.y));
            }
            seg[(j & 1) * 4 + g] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (j & 1) {  // a 64-column block is complete
            const int col0 = nb * BN + (c_begin + j - 1) * 32;
            uint8_t* buf = sb + (nstore % kSoftmaxStoreBufs) * AUX_BUF_BYTES;
            if (lane == 0 && nstore >= kSoftmaxStoreBufs) bulk_wait_group_read<kSoftmaxStoreBufs - 1>();
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
              *reinterpret_cast<uint4*>(buf + lane * 128 + ((jj ^ (lane & 7)) << 4)) = seg[jj];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && col0 < N) {  // a block wholly past N is not stored
              int cc[4];
              aux_coords(col0, mb * BM + q * 32, z1, z2, cc);
              tma_store_4d(&tmap_out, buf, cc[0], cc[1], cc[2], cc[3]);
            }
            if (lane == 0) bulk_commit_group();  // (an empty group for a skipped block keeps the count)
            ++nstore;
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty_bar[acc]);
      }
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
  } else if constexpr (kAux) {
      // dS = escale * P * (dP - D) with P arriving by TMA: pass k (64 columns) of a tile reads
      // buffer k, which lane 0 refills with the next tile's pass k as soon as the warp has read it.
      static_assert(kChunks == 4, "two 64-column passes per warp");
      uint8_t* pb = aux_buf + (warp - 2) * kAuxBufs * AUX_BUF_BYTES;  // buffers 0, 1: P loads
      uint8_t* sb = pb + 2 * AUX_BUF_BYTES;                             // buffers 2, 3: dS stores
      uint64_t* pbar = aux_bar + (warp - 2) * 2;
      int nstore = 0;
      uint32_t pphase[2] = {0u, 0u};
      bool pending[2] = {false, false};
      auto issue_p = [&](int tl, int k) {  // uniform across the warp
        if (tl >= total_tiles) return;
        int z1, z2, mb, nb;
        tile_coords(tl, z1, z2, mb, nb);
        const int col = nb * BN + (c_begin + 2 * k) * 32;
        if (col >= N) return;
        if (lane == 0) {
          fence_proxy_async_smem();  // the warp's reads of this buffer come before the TMA refill
          mbar_arrive_expect_tx(&pbar[k], AUX_BUF_BYTES);
          load_tile<true>(pb + k * AUX_BUF_BYTES, &tmap_aux, &pbar[k], col, mb * BM + q * 32, z1, z2, bd.x_row,
                          bd.x_z1, bd.x_z2);
        }
        pending[k] = true;
      };
      issue_p(blockIdx.x, 0);
      issue_p(blockIdx.x, 1);
      int it = 0;
      bool fail = false;
      for (int tile = blockIdx.x; tile < total_tiles && !fail; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        const bool ok = mbar_wait(&tfull_bar[acc], use & 1, status, 6);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        int z1, z2, mb, nb;
        tile_coords(tile, z1, z2, mb, nb);
        const int64_t row = static_cast<int64_t>(mb) * BM + q * 32 + lane;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
        const int64_t srow = (static_cast<int64_t>(z2) * bd.nz1 + z1) * M + row;
        const float a2 = bd.alpha * ep.escale;
        const float d2 = (row < M ? static_cast<const float*>(ep.rowvec)[srow] : 0.f) * ep.escale;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c = c_begin + 2 * k;
          const int col0 = nb * BN + c * 32;
          if (col0 < N) {  // uniform across the warp
            uint32_t v[64];
            tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), *reinterpret_cast<uint32_t(*)[32]>(v));
            tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32 + 32),
                               *reinterpret_cast<uint32_t(*)[32]>(v + 32));
            const bool okp = mbar_wait(&pbar[k], pphase[k], status, 7);
            pphase[k] ^= 1u;
            pending[k] = false;
            if (!__all_sync(0xffffffffu, okp)) fail = true;
            // The TMA wrote the block with the 128-byte swizzle: row r's 16-byte segment j sits
            // at r * 128 + ((j ^ (r & 7)) << 4), so each thread reads its own row without conflicts.
            uint4 ps[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
              ps[jj] = *reinterpret_cast<const uint4*>(pb + k * AUX_BUF_BYTES + lane * 128 + ((jj ^ (lane & 7)) << 4));
            __syncwarp();
            if (!fail) issue_p(tile + static_cast<int>(gridDim.x), k);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 8; ++g) {  // dS overwrites P in place
              uint32_t* w = reinterpret_cast<uint32_t*>(&ps[g]);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 pf = unpack_bf16x2(w[i]);
                w[i] = pack_bf16x2(pf.x * fmaf(__uint_as_float(v[g * 8 + 2 * i]), a2, -d2),
                                   pf.y * fmaf(__uint_as_float(v[g * 8 + 2 * i + 1]), a2, -d2));
              }
            }
            uint8_t* buf = sb + (nstore & 1) * AUX_BUF_BYTES;
            if (lane == 0 && nstore >= 2) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = ps[j];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              int cc[4];
              aux_coords(col0, mb * BM + q * 32, z1, z2, cc);
              tma_store_4d(&tmap_out, buf, cc[0], cc[1], cc[2], cc[3]);
              bulk_commit_group();
            }
            ++nstore;
          } else if (!fail) {
            issue_p(tile + static_cast<int>(gridDim.x), k);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty_bar[acc]);
      }
      // Copies still in flight finish before the CTA's shared memory goes away (the loads' waits
      // are bounded).
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (pending[k]) mbar_wait(&pbar[k], pphase[k], status, 8);
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
    } else {
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      const bool ok = mbar_wait(&tfull_bar[acc], use & 1, status, 6);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      int z1, z2, mb, nb;
      tile_coords(tile, z1, z2, mb, nb);
      const int64_t out_off = BATCHED ? z1 * bd.out_z1 + z2 * bd.out_z2 : 0;
      const int64_t row = static_cast<int64_t>(mb) * BM + q * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      const int64_t srow = BATCHED ? (static_cast<int64_t>(z2) * bd.nz1 + z1) * M + row : row;
      epilogue_tile<EPI, BATCHED, kChunks>(ep, epi_stage + (warp - 2) * EPI_STAGE_BYTES, lane, row, M, N, nb * BN, c_begin,
                                  t_row, out_off, BATCHED ? bd.alpha : 1.f, srow, nb, sched.num_nb);
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------- CTA-pair kernel
// The same GEMM on 256 x 256 tiles computed by a cluster of two CTAs on two SMs
// (tcgen05 cta_group::2): each CTA loads its 128 rows of A and 128 of the tile's 256 B
// columns, so each SM fills 32 KB of shared memory per 64-deep k-block instead of 48 KB and
// six stages fit where four did; one thread of the even CTA issues M256 N256 K16 MMAs that
// read both CTAs' operands and write 128 accumulator rows into each CTA's tensor memory.
//   barriers: full[s] (even CTA; both CTAs' copies complete on it), empty[s] (each CTA;
//   the MMA commit arrives on both), tfull[acc] (each CTA; multicast commit), tempty[acc]
//   (even CTA; all epilogue threads of both CTAs arrive), drain (even CTA).
//   Every wait is the ordinary CTA-scope try_wait, also on barriers the peer arrives on: what
//   a waiter touches next is shared memory written by TMA and read by the tensor core (async
//   proxy) or tensor memory ordered by the tcgen05 fences around the barrier, never data the
//   peer wrote through the generic proxy. (The 256 epilogue threads spin on a wait for most
//   of a launch; with cluster-scope acquire the step measured 0.5-1 % slower.)
constexpr int PAIR_STAGES = 6;
constexpr int BN_HALF = BN / 2;                               // B columns loaded per CTA
constexpr int PAIR_STAGE_BYTES = A_STAGE_BYTES + BN_HALF * BK * 2;  // 32 KiB
constexpr int PAIR_SMEM_BYTES = PAIR_STAGES * PAIR_STAGE_BYTES + NUM_EPI_WARPS * EPI_STAGE_BYTES + BARRIER_BYTES + 1024;
// Tile band in 256-row pair blocks. Measured on the GPT MLP shape (where the wave model still
// sends GEMMs here): 16 pair-rows 3654 us for the six GEMMs serialised, 12: 3668, 8: 3683, 4: 3724.
constexpr int PAIR_GROUP_M = 16;
static_assert(PAIR_SMEM_BYTES <= 227 * 1024, "shared memory budget (pair kernel)");
static_assert((2 * PAIR_STAGES + 2 * NUM_ACC + 1) * 8 + 4 <= BARRIER_BYTES, "barrier area");

constexpr int kPaceKb = 16;                 // k-blocks between pacing points (16 and 32 measured alike; 64: +0.4 %)
// GeLU' epilogue of the wide kernel: the producer prefetches the tile's Z rows into L2 this many
// k-blocks before the end of the tile's K-loop (map in the second output slot, tma_out bit 2).
constexpr int kAuxPrefetchKb = 16;
constexpr uint64_t kPaceWaitNs = 50000;     // longest pause at one pacing point

// Spins (bounded by limit_ns) until *ctr >= target; a pacing hint, so expiry is not an error.
__device__ __forceinline__ void pace_wait(const unsigned int* ctr, unsigned int target, uint64_t limit_ns) {
  auto read = [&] {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v;
  };
  if (read() >= target) return;
  const uint64_t t0 = global_timer_ns();
  while (read() < target) {
    if (global_timer_ns() - t0 > limit_ns) return;
    __nanosleep(64);
  }
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_c2,
                          int tma_out, int M, int N, int K, EpiParams ep, unsigned int* status, int group,
                          unsigned int* pace) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* epi_stage = smem + PAIR_STAGES * PAIR_STAGE_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(epi_stage + NUM_EPI_WARPS * EPI_STAGE_BYTES);
  uint64_t* empty_bar = full_bar + PAIR_STAGES;
  uint64_t* tfull_bar = empty_bar + PAIR_STAGES;
  uint64_t* tempty_bar = tfull_bar + NUM_ACC;
  uint64_t* drain_bar = tempty_bar + NUM_ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  const int num_mb = (M + 2 * BM - 1) / (2 * BM);
  const int num_nb = (N + BN - 1) / BN;
  const int num_tiles = num_mb * num_nb;
  // group > 0: bands of `group` pair-rows, each walked N-block by N-block (M fastest);
  // group < 0: bands of -group N-blocks, walked pair-row by pair-row (N fastest).
  auto coords = [&](int tile, int& mb, int& nb) {
    if (group > 0) {
      const int group_size = group * num_nb;
      const int g = tile / group_size;
      const int first_mb = g * group;
      const int gsz = min(num_mb - first_mb, group);
      const int in_group = tile - g * group_size;
      mb = first_mb + in_group % gsz;
      nb = in_group / gsz;
    } else {
      const int gn = -group;
      const int group_size = gn * num_mb;
      const int g = tile / group_size;
      const int first_nb = g * gn;
      const int gsz = min(num_nb - first_nb, gn);
      const int in_group = tile - g * group_size;
      nb = first_nb + in_group % gsz;
      mb = in_group / gsz;
    }
  };
  const int num_kb = (K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
#pragma unroll
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
#pragma unroll
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 2 * NUM_EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised in both CTAs before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both CTAs)
      int kiter = 0;
      bool ok = true;
      // Pacing (even CTAs, when pace != null): every kPaceKb k-blocks a pair announces itself on
      // *pace and first waits, for at most kPaceWaitNs, until every pair with a tile in the
      // same round has announced the previous point. Pairs that share operand panels then stay
      // within a few dozen k-blocks of each other and find the panels in L2 instead of
      // re-reading them from DRAM. The wait only delays loads; it is never an error. The host
      // zeroes the counter before the launch.
      const bool pacer = pace != nullptr && rank == 0;
      unsigned int pace_target = 0;  // announcements of all earlier points
      for (int tile = pair, round = 0; tile < num_tiles && ok; tile += num_pairs, ++round) {
        int mb, nb;
        coords(tile, mb, nb);
        const int a_row = mb * 2 * BM + static_cast<int>(rank) * BM;
        const int b_col = nb * BN + static_cast<int>(rank) * BN_HALF;
        const unsigned int active = static_cast<unsigned int>(min(num_pairs, num_tiles - round * num_pairs));
        for (int kb = 0; kb < num_kb; ++kb) {
          if (pacer && kb % kPaceKb == 0) {
            pace_wait(pace, pace_target, kPaceWaitNs);
            atomicAdd(pace, 1u);
            pace_target += active;
          }
          const int s = kiter % PAIR_STAGES;
          const uint32_t parity = ((kiter / PAIR_STAGES) & 1) ^ 1;
          if (!mbar_wait(&empty_bar[s], parity, status, 11)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * PAIR_STAGE_BYTES);
          // K runs backwards in odd rounds: a round starts on the k-blocks that the previous round
          // (which shares its A panels in the band order) touched last, so more of them are in L2.
          const int kbl = (round & 1) ? num_kb - 1 - kb : kb;
          const uint32_t full0 = map_to_cta(&full_bar[s], 0);
          uint8_t* sa = smem + s * PAIR_STAGE_BYTES;
          uint8_t* sb = sa + A_STAGE_BYTES;
          if constexpr (!A_MN) {
            tma_load_2d_pair(sa, &tmap_a, full0, kbl * BK, a_row);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j) tma_load_2d_pair(sa + j * MN_BOX_BYTES, &tmap_a, full0, a_row + j * 64, kbl * BK);
          }
          if constexpr (!B_MN) {
            tma_load_2d_pair(sb, &tmap_b, full0, kbl * BK, b_col);
          } else {
#pragma unroll
            for (int j = 0; j < BN_HALF / 64; ++j)
              tma_load_2d_pair(sb + j * MN_BOX_BYTES, &tmap_b, full0, b_col + j * 64, kbl * BK);
          }
          ++kiter;
        }
      }
      // The even CTA's full barriers count both CTAs' copies: once its last phases have
      // completed (at once on the normal path), no copy of the pair is still in flight.
      if (rank == 0)
        for (int k = max(0, kiter - PAIR_STAGES); k < kiter; ++k)
          mbar_wait(&full_bar[k % PAIR_STAGES], (k / PAIR_STAGES) & 1, status, 12);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA issuer (even CTA)
      constexpr uint32_t kIdesc = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
      int kiter = 0, it = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles; tile += num_pairs, ++it) {
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(&tempty_bar[acc], (use & 1) ^ 1, status, 13)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          const int s = kiter % PAIR_STAGES;
          if (!mbar_wait(&full_bar[s], (kiter / PAIR_STAGES) & 1, status, 14)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * PAIR_STAGE_BYTES);
          const uint32_t b_base = a_base + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t adesc = A_MN ? smem_desc_sw128(a_base + kk * 2048, MN_BOX_BYTES, 1024)
                                        : smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(b_base + kk * 2048, MN_BOX_BYTES, 1024)
                                        : smem_desc_sw128(b_base + kk * 32, 16, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair_mc(&empty_bar[s], 0x3);  // frees stage s in both CTAs
          ++kiter;
        }
        if (!ok) break;
        umma_commit_pair_mc(&tfull_bar[acc], 0x3);  // both halves of the accumulator ready
      }
      umma_commit_pair(drain_bar);
      mbar_wait(drain_bar, 0, status, 15);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int c_begin = ((warp - 2) / 4) * kEpiChunks;
    const CUtensorMap* tm_out = (tma_out & 1) ? &tmap_c : nullptr;  // bulk stores of ep.out / ep.out2
    const CUtensorMap* tm_out2 = (tma_out & 2) ? &tmap_c2 : nullptr;
    int it = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs, ++it) {
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      const bool ok = mbar_wait(&tfull_bar[acc], use & 1, status, 16);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      int mb, nb;
      coords(tile, mb, nb);
      const int64_t row = static_cast<int64_t>(mb) * 2 * BM + rank * BM + q * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epilogue_tile<EPI, false, kEpiChunks, kTmaEpi<EPI>>(ep, epi_stage + (warp - 2) * EPI_STAGE_BYTES, lane, row, M,
                                                          N, nb * BN, c_begin, t_row, 0, 1.f, row, nb, num_nb,
                                                          tm_out, tm_out2);
      tc_fence_before();
      mbar_arrive_cluster(map_to_cta(&tempty_bar[acc], 0));
    }
    if (lane == 0) bulk_wait_group_all();  // the last bulk stores have completed
    __syncwarp();
  }

  // Neither CTA frees tensor memory or leaves (its barriers are targets of the other's
  // arrivals) before both are done.
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// GeLU' epilogue pieces of the wide kernel. load_z_block: the warp's 32 rows x 64 columns of Z
// from row0 / col0 into registers, line-wide (lane: rows row0 + i * 4 + lane / 8, segment
// lane % 8; zeros past M or N), as issue_block_loads for rows that are not remapped.
__device__ __forceinline__ void load_z_block(uint4 (&r8)[8], const EpiParams& ep, int lane, int64_t row0, int col0,
                                             int M, int N) {
  const int64_t r_first = row0 + (lane >> 3);
  const int col = col0 + (lane & 7) * 8;
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(ep.aux) + r_first * ep.ldo + col;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    r8[i] = make_uint4(0, 0, 0, 0);
    if (r_first + i * 4 < M && col < N) r8[i] = *reinterpret_cast<const uint4*>(src + i * 4 * ep.ldo);
  }
}

// D = acc * gelu'(Z) for 32 columns of the lane's row: z[0..3] hold the 32 bf16 Z values and
// receive D; v the 32 accumulator values.
__device__ __forceinline__ void dgelu_32(uint4* z, const uint32_t (&v)[32], int gelu) {
  if (gelu == kGeluTanh) {  // uniform: pairs of elements on the f32x2 path
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t* w = reinterpret_cast<uint32_t*>(&z[g]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const F2 z2 = f2_make(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
        const float2 d2 = f2_split(f2_mul(f2_make(__uint_as_float(v[g * 8 + 2 * i]), __uint_as_float(v[g * 8 + 2 * i + 1])),
                                          gelu_grad_tanh2(z2)));
        w[i] = pack_bf16x2(d2.x, d2.y);
      }
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g)
      z[g] = dgelu_other8(v[g * 8], v[g * 8 + 1], v[g * 8 + 2], v[g * 8 + 3], v[g * 8 + 4], v[g * 8 + 5], v[g * 8 + 6],
                          v[g * 8 + 7], z[g], gelu);
  }
}

// ---------------------------------------------------------------------- wide CTA-pair kernel
// The pair kernel on 256 x 512 tiles: the pair's MMAs cover the tile's two 256-column halves
// with two M256 N256 K16 instructions per K16 step that share the A tile, so each SM receives
// 48 KB of operands per 64-deep k-block (its 128 A rows and two 128-column B chunks) for twice
// the work of the 256 x 256 pair tile: 25 % fewer operand bytes per FLOP into every SM and out
// of L2. The two half accumulators take all 512 tensor-memory columns, so there is one
// accumulator set: the epilogue drains half 0, then half 1, waiting on one full barrier and
// arriving on one empty barrier per half. Both ends of a tile's K-loop are skewed so that a
// drain overlaps MMAs of the other half: over the last WIDE_STAGES k-blocks (their stages stay
// resident) half 0 goes first and is committed on its own, so its drain runs while half 1
// finishes those k-blocks; the next tile's half 0 starts as soon as half 0 is drained and runs
// ahead over the first WIDE_STAGES k-blocks while half 1 is still being drained, then half 1
// catches up on those k-blocks; in between both halves proceed k-block by k-block.
//   barriers: full[s] (even CTA), empty[s] (each CTA), tfull[h] (each CTA; multicast commit),
//   tempty[h] (even CTA; all epilogue threads of both CTAs arrive), drain (even CTA).
constexpr int WIDE_STAGES = 4;
constexpr int WIDE_GROUP_M = 16;  // tile band in pair-rows (measured: 16 beats 8 and 32 on the large MLP)
constexpr int WIDE_BN = 2 * BN;                                 // 512 columns per pair tile
constexpr int WIDE_CHUNK_BYTES = BN_HALF * BK * 2;              // one 128-column B chunk, 16 KiB
constexpr int WIDE_STAGE_BYTES = A_STAGE_BYTES + 2 * WIDE_CHUNK_BYTES;  // 48 KiB
constexpr int WIDE_SMEM_BYTES = WIDE_STAGES * WIDE_STAGE_BYTES + NUM_EPI_WARPS * EPI_STAGE_BYTES + BARRIER_BYTES + 1024;
static_assert(WIDE_SMEM_BYTES <= 227 * 1024, "shared memory budget (wide pair kernel)");
static_assert((2 * WIDE_STAGES + 2 + 2 + 1) * 8 + 4 <= BARRIER_BYTES, "barrier area (wide pair kernel)");

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_wide_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_c2,
                          int tma_out, int M, int N, int K, EpiParams ep, unsigned int* status, int group,
                          unsigned int* pace, int tail_split) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* epi_stage = smem + WIDE_STAGES * WIDE_STAGE_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(epi_stage + NUM_EPI_WARPS * EPI_STAGE_BYTES);
  uint64_t* empty_bar = full_bar + WIDE_STAGES;
  uint64_t* tfull_bar = empty_bar + WIDE_STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  const int num_mb = (M + 2 * BM - 1) / (2 * BM);
  const int num_nb = (N + WIDE_BN - 1) / WIDE_BN;
  const int num_tiles = num_mb * num_nb;
  // group > 0: bands of `group` pair-rows walked along N; group < 0: bands of -group N-blocks
  // walked along M (as in the 256 x 256 pair kernel).
  auto coords = [&](int tile, int& mb, int& nb) {
    if (group > 0) {
      const int group_size = group * num_nb;
      const int g = tile / group_size;
      const int first_mb = g * group;
      const int gsz = min(num_mb - first_mb, group);
      const int in_group = tile - g * group_size;
      mb = first_mb + in_group % gsz;
      nb = in_group / gsz;
    } else {
      const int gn = -group;
      const int group_size = gn * num_mb;
      const int g = tile / group_size;
      const int first_nb = g * gn;
      const int gsz = min(num_nb - first_nb, gn);
      const int in_group = tile - g * group_size;
      nb = first_nb + in_group % gsz;
      mb = in_group / gsz;
    }
  };
  const int num_kb = (K + BK - 1) / BK;
  // Work of round r: wide tile pair + r * num_pairs (half = -1: both halves). With tail_split the
  // last, partial round is split in 256-column half-tiles, one per pair (pairs 2i and 2i + 1 take
  // the two halves of the round's i-th tile), so that it takes about half a round.
  const int rounds_full = (num_tiles + num_pairs - 1) / num_pairs - (tail_split ? 1 : 0);
  const int tail_tiles = num_tiles - rounds_full * num_pairs;
  auto work = [&](int round, int& tile, int& half) -> bool {
    if (round < rounds_full) {
      tile = pair + round * num_pairs;
      half = -1;
      return tile < num_tiles;
    }
    if (!tail_split || round > rounds_full || pair >= 2 * tail_tiles) return false;
    tile = rounds_full * num_pairs + (pair >> 1);
    half = pair & 1;
    return true;
  };

  if (warp == 0 && lane == 0) {
#pragma unroll
    for (int s = 0; s < WIDE_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar[0], 1);
    mbar_init(&tfull_bar[1], 1);
    mbar_init(&tempty_bar[0], 2 * NUM_EPI_THREADS);
    mbar_init(&tempty_bar[1], 2 * NUM_EPI_THREADS);
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised in both CTAs before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both CTAs)
      int kiter = 0;
      bool ok = true;
      const bool pacer = pace != nullptr && rank == 0;  // pacing as in the 256 x 256 pair kernel
      // A panels are reused by every tile of a band: their lines are kept in L2 before others
      // (DRAM reads per large-MLP step 37.8 -> 36.3 GB; marking B evict-first as well re-read
      // B: 49 GB)
      const uint64_t pol_a = l2_policy_evict_last();
      unsigned int pace_target = 0;
      int tile, half;
      for (int round = 0; ok && work(round, tile, half); ++round) {
        int mb, nb;
        coords(tile, mb, nb);
        const int a_row = mb * 2 * BM + static_cast<int>(rank) * BM;
        const unsigned int active = static_cast<unsigned int>(
            round < rounds_full ? min(num_pairs, num_tiles - round * num_pairs) : 2 * tail_tiles);
        const uint32_t stage_tx = half < 0 ? 2 * WIDE_STAGE_BYTES : 2 * (A_STAGE_BYTES + WIDE_CHUNK_BYTES);
        for (int kb = 0; kb < num_kb; ++kb) {
          if constexpr (EPI == kEpiDGelu) {
            // Z of this CTA's 128 output rows into L2 some k-blocks before the epilogue reads it
            if ((tma_out & 4) && kb == max(0, num_kb - kAuxPrefetchKb))
              for (int j = (half == 1 ? 4 : 0); j < (half == 0 ? 4 : 8); ++j)
                tma_prefetch_l2_2d(&tmap_c2, nb * WIDE_BN + j * 64, a_row);
          }
          if (pacer && kb % kPaceKb == 0) {
            pace_wait(pace, pace_target, kPaceWaitNs);
            atomicAdd(pace, 1u);
            pace_target += active;
          }
          const int s = kiter % WIDE_STAGES;
          const uint32_t parity = ((kiter / WIDE_STAGES) & 1) ^ 1;
          if (!mbar_wait(&empty_bar[s], parity, status, 31)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], stage_tx);
          const int kbl = (round & 1) ? num_kb - 1 - kb : kb;  // K backwards in odd rounds (as above)
          const uint32_t full0 = map_to_cta(&full_bar[s], 0);
          uint8_t* sa = smem + s * WIDE_STAGE_BYTES;
          uint8_t* sb = sa + A_STAGE_BYTES;
          if constexpr (!A_MN) {
            tma_load_2d_pair_hint(sa, &tmap_a, full0, kbl * BK, a_row, pol_a);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j) tma_load_2d_pair_hint(sa + j * MN_BOX_BYTES, &tmap_a, full0, a_row + j * 64, kbl * BK, pol_a);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // this CTA's 128 columns of each 256-column half
            if (half >= 0 && h != half) continue;
            const int b_col = nb * WIDE_BN + h * BN + static_cast<int>(rank) * BN_HALF;
            uint8_t* sbh = sb + h * WIDE_CHUNK_BYTES;
            if constexpr (!B_MN) {
              tma_load_2d_pair(sbh, &tmap_b, full0, kbl * BK, b_col);
            } else {
#pragma unroll
              for (int j = 0; j < BN_HALF / 64; ++j)
                tma_load_2d_pair(sbh + j * MN_BOX_BYTES, &tmap_b, full0, b_col + j * 64, kbl * BK);
            }
          }
          ++kiter;
        }
      }
      // The even CTA's full barriers count both CTAs' copies: once its last phases have
      // completed (at once on the normal path), no copy of the pair is still in flight.
      if (rank == 0)
        for (int k = max(0, kiter - WIDE_STAGES); k < kiter; ++k)
          mbar_wait(&full_bar[k % WIDE_STAGES], (k / WIDE_STAGES) & 1, status, 32);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA issuer (even CTA)
      constexpr uint32_t kIdesc = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
      // The four K16 MMAs of k-block kb (stage s) into half h of the accumulator.
      auto issue_half = [&](int s, int kb, int h) {
        const uint32_t a_base = smem_u32(smem + s * WIDE_STAGE_BYTES);
        const uint32_t bh = a_base + A_STAGE_BYTES + h * WIDE_CHUNK_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t adesc = A_MN ? smem_desc_sw128(a_base + kk * 2048, MN_BOX_BYTES, 1024)
                                      : smem_desc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bdesc = B_MN ? smem_desc_sw128(bh + kk * 2048, MN_BOX_BYTES, 1024)
                                      : smem_desc_sw128(bh + kk * 32, 16, 1024);
          umma_bf16_pair(tmem_base + static_cast<uint32_t>(h * BN), adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
        }
      };
      int kiter = 0, it = 0;
      bool ok = true;
      int tile, half;
      for (; ok && work(it, tile, half); ++it) {
        const uint32_t prev = static_cast<uint32_t>(it & 1) ^ 1;  // phase of the previous tile's drain
        if (half >= 0) {
          // A half-tile of the split last round: only accumulator half `half`, committed on its
          // full barrier (the other half's barriers see no more phases).
          if (!mbar_wait(&tempty_bar[half], prev, status, 34)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < num_kb; ++kb) {
            const int s = kiter % WIDE_STAGES;
            if (!mbar_wait(&full_bar[s], (kiter / WIDE_STAGES) & 1, status, 33)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_half(s, kb, half);
            umma_commit_pair_mc(&empty_bar[s], 0x3);
            ++kiter;
          }
          if (!ok) break;
          umma_commit_pair_mc(&tfull_bar[half], 0x3);
          continue;
        }
        // Half 0 runs ahead over the first `lead` k-blocks, while the epilogue may still be
        // draining half 1 of the previous tile; those stages stay resident until half 1 has
        // used them too, then each is freed. Over the last `tail` k-blocks half 0 goes first
        // again and is committed on its own, so that its drain overlaps half 1's last MMAs.
        const int lead = min(WIDE_STAGES, num_kb);
        const int tail = min(WIDE_STAGES, num_kb - lead);
        if (!mbar_wait(&tempty_bar[0], prev, status, 34)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < lead; ++kb) {
          const int k = kiter + kb;
          if (!mbar_wait(&full_bar[k % WIDE_STAGES], (k / WIDE_STAGES) & 1, status, 33)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_half(k % WIDE_STAGES, kb, 0);
        }
        if (!ok) break;
        if (tail == 0) umma_commit_pair_mc(&tfull_bar[0], 0x3);  // half 0 complete (num_kb <= lead)
        if (!mbar_wait(&tempty_bar[1], prev, status, 34)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < lead; ++kb) {
          const int s = (kiter + kb) % WIDE_STAGES;
          issue_half(s, kb, 1);
          umma_commit_pair_mc(&empty_bar[s], 0x3);  // frees stage s in both CTAs
        }
        kiter += lead;
        for (int kb = lead; kb < num_kb - tail; ++kb) {
          const int s = kiter % WIDE_STAGES;
          if (!mbar_wait(&full_bar[s], (kiter / WIDE_STAGES) & 1, status, 33)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_half(s, kb, 0);
          issue_half(s, kb, 1);
          umma_commit_pair_mc(&empty_bar[s], 0x3);
          ++kiter;
        }
        if (!ok) break;
        if (tail > 0) {
          for (int j = 0; j < tail; ++j) {
            const int k = kiter + j;
            if (!mbar_wait(&full_bar[k % WIDE_STAGES], (k / WIDE_STAGES) & 1, status, 33)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_half(k % WIDE_STAGES, num_kb - tail + j, 0);
          }
          if (!ok) break;
          umma_commit_pair_mc(&tfull_bar[0], 0x3);  // half 0 of both CTAs' accumulators ready
          for (int j = 0; j < tail; ++j) {
            const int s = (kiter + j) % WIDE_STAGES;
            issue_half(s, num_kb - tail + j, 1);
            umma_commit_pair_mc(&empty_bar[s], 0x3);
          }
          kiter += tail;
        }
        umma_commit_pair_mc(&tfull_bar[1], 0x3);  // half 1 ready
      }
      umma_commit_pair(drain_bar);
      mbar_wait(drain_bar, 0, status, 35);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int c_begin = ((warp - 2) / 4) * kEpiChunks;
    const CUtensorMap* tm_out = (tma_out & 1) ? &tmap_c : nullptr;  // bulk stores of ep.out / ep.out2
    const CUtensorMap* tm_out2 = (tma_out & 2) ? &tmap_c2 : nullptr;
    int it = 0;
    bool ok = true;
    if constexpr (EPI == kEpiDGelu) {
      // The warp's four 64-column passes of a tile (two per half) are pipelined on Z: the next
      // pass's Z is loaded into registers while this one is computed, and the tile's first pass
      // is loaded before its accumulator is ready, so no pass waits for its Z. Stores by bulk
      // tensor copies (tm_out is always set for this kind).
      uint8_t* buf = epi_stage + (warp - 2) * EPI_STAGE_BYTES;
      int tile, half;
      for (; ok && work(it, tile, half); ++it) {
        int mb, nb;
        coords(tile, mb, nb);
        const int64_t row0 = static_cast<int64_t>(mb) * 2 * BM + rank * BM + q * 32;
        auto pass_col = [&](int p) { return nb * WIDE_BN + (p >> 1) * BN + (c_begin + 2 * (p & 1)) * 32; };
        const int h_first = half < 0 ? 0 : half, h_last = half < 0 ? 1 : half;  // a half-tile: one half
        uint4 r8[8];
        load_z_block(r8, ep, lane, row0, pass_col(2 * h_first), M, N);
#pragma unroll 1
        for (int h = h_first; h <= h_last; ++h) {
          ok = __all_sync(0xffffffffu, mbar_wait(&tfull_bar[h], static_cast<uint32_t>(it & 1), status, 36));
          if (!ok) break;
          tc_fence_after();
          const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * BN);
#pragma unroll 1
          for (int k = 0; k < 2; ++k) {
            const int p = 2 * h + k;
            const int col0 = pass_col(p);
            uint4 zs[8];
            buf_acquire(lane);  // the previous pass's bulk store has read the buffer
            transpose_block(buf, r8, zs, lane);
            if (p < 2 * h_last + 1) load_z_block(r8, ep, lane, row0, pass_col(p + 1), M, N);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>((c_begin + 2 * k + j) * 32), v);
              tmem_ld_wait();
              dgelu_32(&zs[4 * j], v, ep.gelu);
            }
            if (col0 < N) store_tma(buf, zs, lane, tm_out, col0, static_cast<int>(row0));
          }
          tc_fence_before();
          mbar_arrive_cluster(map_to_cta(&tempty_bar[h], 0));
        }
      }
    } else {
      int tile, half;
      for (; ok && work(it, tile, half); ++it) {
        int mb, nb;
        coords(tile, mb, nb);
        const int64_t row = static_cast<int64_t>(mb) * 2 * BM + rank * BM + q * 32 + lane;
#pragma unroll 1
        for (int h = (half < 0 ? 0 : half); h <= (half < 0 ? 1 : half); ++h) {
          ok = __all_sync(0xffffffffu, mbar_wait(&tfull_bar[h], static_cast<uint32_t>(it & 1), status, 36));
          if (!ok) break;
          tc_fence_after();
          const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * BN);
          epilogue_tile<EPI, false, kEpiChunks, kTmaEpi<EPI>>(ep, epi_stage + (warp - 2) * EPI_STAGE_BYTES, lane, row,
                                                              M, N, nb * WIDE_BN + h * BN, c_begin, t_row, 0, 1.f, row,
                                                              2 * nb + h, 2 * num_nb, tm_out, tm_out2);
          tc_fence_before();
          mbar_arrive_cluster(map_to_cta(&tempty_bar[h], 0));
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();  // the last bulk stores have completed
    __syncwarp();
  }

  // Neither CTA frees tensor memory or leaves (its barriers are targets of the other's
  // arrivals) before both are done.
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  *fn = g_encode;
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with row stride ld elements.
cudaError_t make_tmap(CUtensorMap* map, const Operand& op, uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  cudaError_t e = get_encode(&encode);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(op.cols), static_cast<cuuint64_t>(op.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(op.ld) * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(op.ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor maps of the pair kernels' outputs for bulk tensor stores: 32-row boxes of 128 bytes
// (64 bf16 or 32 fp32 columns), 128-byte swizzle, matching the epilogue's staging layout. flags
// bit 0: ep.out has a map in c; bit 1: ep.out2 has one in c2. Outputs whose rows are remapped,
// and the kinds that read or reduce in place, keep the per-thread stores.
struct OutMaps {
  CUtensorMap c, c2;
  int flags = 0;
};

cudaError_t make_out_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool f32,
                         uint32_t box_rows = 32) {
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  cudaError_t e = get_encode(&encode);
  if (e != cudaSuccess) return e;
  const cuuint64_t elt = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                      const_cast<void*>(ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_out_maps(OutMaps* om, EpiKind epi, const EpiParams& ep, int64_t M, int64_t N, bool wide) {
  om->flags = 0;
  const bool kind_ok = epi == kEpiStore || epi == kEpiStoreF32 || epi == kEpiGelu || (wide && epi == kEpiDGelu);
  if (!kind_ok || ep.remap.enabled) return cudaSuccess;
  const bool f32 = epi == kEpiStoreF32;
  const int64_t elt = f32 ? 4 : 2;
  // A tensor map wants a 16-byte aligned base and a row stride that is a multiple of 16 bytes.
  auto fits = [&](const void* p) {
    return p != nullptr && reinterpret_cast<uintptr_t>(p) % 16 == 0 && (ep.ldo * elt) % 16 == 0 && ep.ldo >= N;
  };
  if (fits(ep.out)) {
    cudaError_t e = make_out_map(&om->c, ep.out, M, N, ep.ldo, f32);
    if (e != cudaSuccess) return e;
    om->flags |= 1;
  }
  if (epi == kEpiGelu && fits(ep.out2)) {
    cudaError_t e = make_out_map(&om->c2, ep.out2, M, N, ep.ldo, false);
    if (e != cudaSuccess) return e;
    om->flags |= 2;
  }
  if (epi == kEpiDGelu && fits(ep.aux)) {  // Z, for the producer's L2 prefetch (128-row boxes)
    cudaError_t e = make_out_map(&om->c2, ep.aux, M, N, ep.ldo, false, BM);
    if (e != cudaSuccess) return e;
    om->flags |= 4;
  }
  // GeLU (both pair kernels) and GeLU' (the wide one) compile the bulk-store path alone: every
  // output they write needs its map (the API's shape and alignment checks guarantee it).
  if (epi == kEpiGelu && ((ep.out && !(om->flags & 1)) || !(om->flags & 2))) return cudaErrorInvalidValue;
  if (wide && epi == kEpiDGelu && !(om->flags & 1)) return cudaErrorInvalidValue;
  return cudaSuccess;
}

template <bool A_MN, bool B_MN, int EPI, bool BATCHED = false, int BN_T = 256>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, const EpiParams& ep,
                   cudaStream_t stream, const DeviceCtx& ctx, const BatchDev& bd = BatchDev{},
                   const CUtensorMap* taux = nullptr, const CUtensorMap* tout = nullptr) {
  auto kernel = gemm_bf16_kernel<A_MN, B_MN, EPI, BATCHED, BN_T>;
  constexpr int kSmem = OneSm<BN_T, aux_bufs<EPI, BATCHED>()>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int64_t tiles = static_cast<int64_t>((M + BM - 1) / BM) * ((N + BN_T - 1) / BN_T);
  if (BATCHED) tiles *= static_cast<int64_t>(bd.nz1) * bd.nz2;
  if (tiles > INT32_MAX) return cudaErrorInvalidValue;
  const int grid = tiles < ctx.num_sms ? static_cast<int>(tiles) : ctx.num_sms;
  kernel<<<grid, NUM_THREADS, kSmem, stream>>>(ta, tb, taux ? *taux : ta, tout ? *tout : ta, M, N, K, ep, ctx.status,
                                               bd);
  return cudaGetLastError();
}

// Pacing counters of the pair kernel: a small pool handed out round-robin so that launches
// in flight on different streams use different counters; each is zeroed on the launch's
// stream before the launch. Pacing is on unless tpmlp_set_gemm_variant turned it off.
__device__ unsigned int g_pace_counters[64];

unsigned int* next_pace_counter() {
  if (!g_pair_pacing.load(std::memory_order_relaxed)) return nullptr;
  static std::atomic<unsigned int> next{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return nullptr;
  static unsigned int* base[16] = {};
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_pace_counters) != cudaSuccess) return nullptr;
      base[dev] = static_cast<unsigned int*>(p);
    }
  }
  return base[dev] + (next.fetch_add(1) % 64);
}

// Tile-order band of the pair kernels (see gemm_bf16_pair_kernel): PAIR_GROUP_M pair-rows for
// 256 x 256 tiles and WIDE_GROUP_M for 256 x 512 tiles, unless tpmlp_set_gemm_variant chose
// another band.
int pair_group(bool wide = false) {
  const int g = g_pair_group.load(std::memory_order_relaxed);
  return g != 0 ? g : (wide ? WIDE_GROUP_M : PAIR_GROUP_M);
}

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const OutMaps& om, int M, int N, int K,
                        const EpiParams& ep, cudaStream_t stream, const DeviceCtx& ctx) {
  auto kernel = gemm_bf16_pair_kernel<A_MN, B_MN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PAIR_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t tiles = static_cast<int64_t>((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // The persistent grid (and the pacing, which waits for every pair of a round) assumes all
  // pairs are resident at once: no more pairs than the device runs concurrently. Every pair
  // instantiation has the same threads and shared memory, so one query per device serves all.
  static int resident_pairs[16] = {};
  static std::mutex mu;
  int max_pairs = ctx.num_sms / 2;
  if (ctx.device >= 0 && ctx.device < 16) {
    std::lock_guard<std::mutex> lock(mu);
    if (resident_pairs[ctx.device] == 0) {
      cfg.gridDim = dim3(2, 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) n = ctx.num_sms / 2;
      resident_pairs[ctx.device] = n < ctx.num_sms / 2 ? n : ctx.num_sms / 2;
    }
    max_pairs = resident_pairs[ctx.device];
  }
  const int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  unsigned int* pace = next_pace_counter();
  if (pace) {
    e = cudaMemsetAsync(pace, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, om.c, om.c2, om.flags, M, N, K, ep, ctx.status, pair_group(), pace);
}

// The wide pair kernel, launched like the 256 x 256 pair kernel (persistent grid of resident pairs,
// pacing counter zeroed on the stream).
template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_wide(const CUtensorMap& ta, const CUtensorMap& tb, const OutMaps& om, int M, int N, int K,
                        const EpiParams& ep, cudaStream_t stream, const DeviceCtx& ctx) {
  auto kernel = gemm_bf16_wide_kernel<A_MN, B_MN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WIDE_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t tiles = static_cast<int64_t>((M + 2 * BM - 1) / (2 * BM)) * ((N + WIDE_BN - 1) / WIDE_BN);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = WIDE_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int resident_pairs[16] = {};
  static std::mutex mu;
  int max_pairs = ctx.num_sms / 2;
  if (ctx.device >= 0 && ctx.device < 16) {
    std::lock_guard<std::mutex> lock(mu);
    if (resident_pairs[ctx.device] == 0) {
      cfg.gridDim = dim3(2, 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) n = ctx.num_sms / 2;
      resident_pairs[ctx.device] = n < ctx.num_sms / 2 ? n : ctx.num_sms / 2;
    }
    max_pairs = resident_pairs[ctx.device];
  }
  // A last round with at most half the pairs busy is split into half-tiles (one per pair).
  int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
  int tail_split = 0;
  const int64_t waves = (tiles + max_pairs - 1) / max_pairs, tail = tiles - (waves - 1) * max_pairs;
  if (2 * tail <= max_pairs) {
    tail_split = 1;
    pairs = static_cast<int>(waves > 1 ? max_pairs : 2 * tail);
  }
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  unsigned int* pace = next_pace_counter();
  if (pace) {
    e = cudaMemsetAsync(pace, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, om.c, om.c2, om.flags, M, N, K, ep, ctx.status, pair_group(true),
                            pace, tail_split);
}

// The pair kernel (256 x 512 tiles if kWide, else 256 x 256) for one operand layout and epilogue.
template <bool kWide>
cudaError_t dispatch_pair(bool a_mn, bool b_mn, EpiKind epi, const CUtensorMap& ta, const CUtensorMap& tb,
                          const OutMaps& om, int m, int n, int k, const EpiParams& ep, cudaStream_t stream,
                          const DeviceCtx& ctx) {
#define TPMLP_PAIR_LAUNCH(AM, BMN, E)                                               \
  return kWide ? launch_wide<AM, BMN, E>(ta, tb, om, m, n, k, ep, stream, ctx)     \
               : launch_pair<AM, BMN, E>(ta, tb, om, m, n, k, ep, stream, ctx)
  if (!a_mn && b_mn) {
    if (epi == kEpiGelu) TPMLP_PAIR_LAUNCH(false, true, kEpiGelu);
    if (epi == kEpiStore) TPMLP_PAIR_LAUNCH(false, true, kEpiStore);
    if (epi == kEpiStoreF32) TPMLP_PAIR_LAUNCH(false, true, kEpiStoreF32);
    if (epi == kEpiDropoutResidual) TPMLP_PAIR_LAUNCH(false, true, kEpiDropoutResidual);
  } else if (!a_mn && !b_mn) {
    if (epi == kEpiDGelu) TPMLP_PAIR_LAUNCH(false, false, kEpiDGelu);
    if (epi == kEpiStore) TPMLP_PAIR_LAUNCH(false, false, kEpiStore);
    if (epi == kEpiStoreRowDot) TPMLP_PAIR_LAUNCH(false, false, kEpiStoreRowDot);
    if (epi == kEpiStoreF32) TPMLP_PAIR_LAUNCH(false, false, kEpiStoreF32);
  } else if (a_mn && b_mn) {
    if (epi == kEpiStoreF32) TPMLP_PAIR_LAUNCH(true, true, kEpiStoreF32);
    if (epi == kEpiAccumF32) TPMLP_PAIR_LAUNCH(true, true, kEpiAccumF32);
  }
#undef TPMLP_PAIR_LAUNCH
  return cudaErrorNotSupported;
}

// Kernel for the plain GEMMs (tpmlp_set_gemm_variant): 0 the single-SM kernel; 1 SM pairs with
// 256 x 512 or 256 x 256 tiles, whichever prefer_wide rates faster; 2 SM pairs with 256 x 256
// tiles only; 3 SM pairs with 256 x 512 tiles only.
int pair_kernel_choice() { return g_pair_kernel.load(std::memory_order_relaxed); }

// Whether 256 x 512 tiles beat 256 x 256 tiles for one GEMM, by a model of the persistent launch:
// its waves of tiles over the resident pairs (a partial last wave costs a full one); a 256 x 512
// wave costs 2 x (u + e / K) of a 256 x 256 one. u is the gain of 25 % fewer operand bytes per
// FLOP, e / K the epilogue that the single accumulator set leaves exposed once per wide tile, in
// k-values of main loop. Fitted per epilogue kind on GB300 (serialised launch times of both tile
// shapes at K = 4096-32768: the three MLP shapes and the attention projections): fp32 stores
// (weight gradients, both operands MN-major) u 0.875, e 40; bf16 stores u 0.905, e 180; GeLU
// u 0.92, e 200; GeLU' (reads Z, pipelined) u 0.87, e 570; the row-dot epilogue u 0.91, e 450;
// dropout + residual (per-thread hash, residual loads, remapped stores) u 0.91, e 2000 (the SP
// block's FC2: 602 us on 256 x 256 tiles, 618 us on split 256 x 512 ones). The fp32
// read-add-write epilogue is not fitted and keeps the earlier, cautious u 0.91 with e 400.
bool prefer_wide(int64_t M, int64_t N, int64_t K, EpiKind epi, int pairs) {
  const int64_t mb = (M + 2 * BM - 1) / (2 * BM);
  const int64_t t256 = mb * ((N + BN - 1) / BN), t512 = mb * ((N + WIDE_BN - 1) / WIDE_BN);
  const int64_t w256 = (t256 + pairs - 1) / pairs, w512 = (t512 + pairs - 1) / pairs;
  double u = 0.905, e = 180.0;  // bf16 stores
  switch (epi) {
    case kEpiStoreF32: u = 0.875; e = 40.0; break;
    case kEpiGelu: u = 0.92; e = 200.0; break;
    case kEpiDGelu: u = 0.87; e = 570.0; break;
    case kEpiStoreRowDot: u = 0.91; e = 450.0; break;
    case kEpiDropoutResidual: u = 0.91; e = 2000.0; break;
    case kEpiAccumF32: u = 0.91; e = 400.0; break;
    default: break;
  }
  const double unit = u + e / static_cast<double>(K);
  // The wide kernel splits a last round that would keep at most half the pairs busy into
  // half-tiles: that round then costs about one 256 x 256 wave.
  const int64_t tail = t512 - (w512 - 1) * pairs;
  const double wide = 2 * tail <= pairs ? 2.0 * unit * static_cast<double>(w512 - 1) + 1.0
                                        : 2.0 * unit * static_cast<double>(w512);
  return wide < static_cast<double>(w256);
}

// 4-D bf16 tensor map over a batched operand: dimension 0 is the contiguous column index; the
// row index and the two batch indices take dimensions 1..3 in order of increasing stride.
// box_inner x box_row elements are copied per load (one row slab of one batch index).
cudaError_t make_tmap_batched(CUtensorMap* map, const BatchedOperand& op, int64_t nz1, int64_t nz2,
                              uint32_t box_inner, uint32_t box_row, int* slot_row, int* slot_z1, int* slot_z2) {
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  cudaError_t e = get_encode(&encode);
  if (e != cudaSuccess) return e;
  struct D { int64_t extent, stride; int id; };
  // extent-1 batch dimensions get a stride past everything else, so they sort last
  int64_t far = (op.rows * op.ld + (nz1 - 1) * op.z1_stride + (nz2 - 1) * op.z2_stride + 1) * 2;
  far = (far + 7) / 8 * 8;  // a multiple of 8 elements, i.e. of 16 bytes, like every TMA stride
  D d[3] = {{op.rows, op.ld, 0}, {nz1, nz1 > 1 ? op.z1_stride : far, 1}, {nz2, nz2 > 1 ? op.z2_stride : far, 2}};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (d[j].stride < d[i].stride || (d[j].stride == d[i].stride && d[j].id < d[i].id)) {
        D t = d[i]; d[i] = d[j]; d[j] = t;
      }
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(op.cols), 0, 0, 0};
  cuuint64_t strides[3];
  cuuint32_t box[4] = {box_inner, 1, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 3; ++i) {
    dims[i + 1] = static_cast<cuuint64_t>(d[i].extent);
    strides[i] = static_cast<cuuint64_t>(d[i].stride) * 2;
    if (d[i].id == 0) { box[i + 1] = box_row; *slot_row = i + 1; }
    if (d[i].id == 1) *slot_z1 = i + 1;
    if (d[i].id == 2) *slot_z2 = i + 1;
  }
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(op.ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

void set_gemm_variant(int pair_kernel, int pair_pacing, int pair_group) {
  g_pair_kernel.store(pair_kernel, std::memory_order_relaxed);
  g_pair_pacing.store(pair_pacing, std::memory_order_relaxed);
  g_pair_group.store(pair_group, std::memory_order_relaxed);
}

cudaError_t gemm_bf16_tc(int64_t M, int64_t N, int64_t K, const Operand& a, const Operand& b, EpiKind epi,
                         const EpiParams& ep, cudaStream_t stream, const DeviceCtx& ctx) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaErrorInvalidValue;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return cudaErrorInvalidValue;
  // The stored shapes must match the contraction.
  if (a.mn_major ? (a.rows != K || a.cols != M) : (a.rows != M || a.cols != K)) return cudaErrorInvalidValue;
  if (b.mn_major ? (b.rows != K || b.cols != N) : (b.rows != N || b.cols != K)) return cudaErrorInvalidValue;
  const int choice = pair_kernel_choice();
  const bool pair = choice >= 1 && ctx.num_sms >= 2;
  const bool wide = pair && (choice == 3 || (choice == 1 && prefer_wide(M, N, K, epi, ctx.num_sms / 2)));
  CUtensorMap ta, tb;
  cudaError_t e = make_tmap(&ta, a, 64, a.mn_major ? BK : BM);
  if (e != cudaSuccess) return e;
  e = make_tmap(&tb, b, 64, b.mn_major ? BK : (pair ? BN_HALF : BN));
  if (e != cudaSuccess) return e;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (pair) {
    if (epi == kEpiDropoutResidual && N % 32 != 0) return cudaErrorInvalidValue;
    OutMaps om;
    e = make_out_maps(&om, epi, ep, M, N, wide);
    if (e != cudaSuccess) return e;
    return wide ? dispatch_pair<true>(a.mn_major, b.mn_major, epi, ta, tb, om, m, n, k, ep, stream, ctx)
                : dispatch_pair<false>(a.mn_major, b.mn_major, epi, ta, tb, om, m, n, k, ep, stream, ctx);
  }
  if (!a.mn_major && b.mn_major) {
    if (epi == kEpiGelu) return launch<false, true, kEpiGelu>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiStore) return launch<false, true, kEpiStore>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiStoreF32) return launch<false, true, kEpiStoreF32>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiDropoutResidual) {
      if (N % 32 != 0) return cudaErrorInvalidValue;
      return launch<false, true, kEpiDropoutResidual>(ta, tb, m, n, k, ep, stream, ctx);
    }
  } else if (!a.mn_major && !b.mn_major) {
    if (epi == kEpiDGelu) return launch<false, false, kEpiDGelu>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiStore) return launch<false, false, kEpiStore>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiStoreRowDot) return launch<false, false, kEpiStoreRowDot>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiStoreF32) return launch<false, false, kEpiStoreF32>(ta, tb, m, n, k, ep, stream, ctx);
  } else if (a.mn_major && b.mn_major) {
    if (epi == kEpiStoreF32) return launch<true, true, kEpiStoreF32>(ta, tb, m, n, k, ep, stream, ctx);
    if (epi == kEpiAccumF32) return launch<true, true, kEpiAccumF32>(ta, tb, m, n, k, ep, stream, ctx);
  }
  return cudaErrorNotSupported;
}

cudaError_t gemm_bf16_tc_batched(int64_t M, int64_t N, int64_t K, const BatchedOperand& a, const BatchedOperand& b,
                                 const BatchSpec& bs, EpiKind epi, const EpiParams& ep, cudaStream_t stream,
                                 const DeviceCtx& ctx) {
  if (M <= 0 || N <= 0 || K <= 0 || bs.nz1 <= 0 || bs.nz2 <= 0) return cudaErrorInvalidValue;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || bs.nz1 > INT32_MAX || bs.nz2 > INT32_MAX)
    return cudaErrorInvalidValue;
  if (a.mn_major ? (a.rows != K || a.cols != M) : (a.rows != M || a.cols != K)) return cudaErrorInvalidValue;
  if (b.mn_major ? (b.rows != K || b.cols != N) : (b.rows != N || b.cols != K)) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  BatchDev bd{};
  bd.nz1 = static_cast<int>(bs.nz1);
  bd.nz2 = static_cast<int>(bs.nz2);
  bd.out_z1 = bs.out_z1;
  bd.out_z2 = bs.out_z2;
  bd.alpha = bs.alpha;
  cudaError_t e = make_tmap_batched(&ta, a, bs.nz1, bs.nz2, 64, a.mn_major ? BK : BM, &bd.a_row, &bd.a_z1, &bd.a_z2);
  if (e != cudaSuccess) return e;
  e = make_tmap_batched(&tb, b, bs.nz1, bs.nz2, 64, b.mn_major ? BK : BN, &bd.b_row, &bd.b_z1, &bd.b_z2);
  if (e != cudaSuccess) return e;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  // N <= 128 with B stored MN-major (the head_dim-wide P V, P^T dO, dS K, dS^T Q): 128-wide tiles,
  // no padded half. An MN-major B is loaded in 64-column boxes, so its tensor map is the same.
  if (N <= 128 && b.mn_major && epi == kEpiStore) {
    if (!a.mn_major) return launch<false, true, kEpiStore, true, 128>(ta, tb, m, n, k, ep, stream, ctx, bd);
    return launch<true, true, kEpiStore, true, 128>(ta, tb, m, n, k, ep, stream, ctx, bd);
  }
  if (!a.mn_major && !b.mn_major && epi == kEpiStoreF32)
    return launch<false, false, kEpiStoreF32, true>(ta, tb, m, n, k, ep, stream, ctx, bd);
  if (!a.mn_major && !b.mn_major && epi == kEpiRowStats)
    return launch<false, false, kEpiRowStats, true>(ta, tb, m, n, k, ep, stream, ctx, bd);
  if (!a.mn_major && !b.mn_major && epi == kEpiSoftmax) {
    // P is written by TMA stores in 64-column x 32-row blocks.
    CUtensorMap tout;
    const BatchedOperand po{ep.out, M, N, ep.ldo, bs.out_z1, bs.out_z2, false};
    e = make_tmap_batched(&tout, po, bs.nz1, bs.nz2, 64, 32, &bd.x_row, &bd.x_z1, &bd.x_z2);
    if (e != cudaSuccess) return e;
    return launch<false, false, kEpiSoftmax, true>(ta, tb, m, n, k, ep, stream, ctx, bd, nullptr, &tout);
  }
  if (!a.mn_major && !b.mn_major && epi == kEpiSoftmaxGrad) {
    // P (the aux operand, laid out like the output) is read by TMA in 64-column x 32-row blocks.
    // dS, laid out like P, is written by TMA stores through the same block shape.
    CUtensorMap taux, tout;
    const BatchedOperand pa{ep.aux, M, N, ep.ldo, bs.out_z1, bs.out_z2, false};
    e = make_tmap_batched(&taux, pa, bs.nz1, bs.nz2, 64, 32, &bd.x_row, &bd.x_z1, &bd.x_z2);
    if (e != cudaSuccess) return e;
    const BatchedOperand po{ep.out, M, N, ep.ldo, bs.out_z1, bs.out_z2, false};
    e = make_tmap_batched(&tout, po, bs.nz1, bs.nz2, 64, 32, &bd.x_row, &bd.x_z1, &bd.x_z2);
    if (e != cudaSuccess) return e;
    return launch<false, false, kEpiSoftmaxGrad, true>(ta, tb, m, n, k, ep, stream, ctx, bd, &taux, &tout);
  }
  if (!a.mn_major && b.mn_major && epi == kEpiStore)
    return launch<false, true, kEpiStore, true>(ta, tb, m, n, k, ep, stream, ctx, bd);
  if (a.mn_major && b.mn_major && epi == kEpiStore)
    return launch<true, true, kEpiStore, true>(ta, tb, m, n, k, ep, stream, ctx, bd);
  return cudaErrorNotSupported;
}

}  // namespace tpmlp
