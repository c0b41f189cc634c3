// Memory-bound kernels of the sequence-parallel MLP block ("Megatron-SP 机制", section
// "通信插在层内什么位置？"): LayerNorm on [b, s/t, h] shards, the all-gather g that turns
// shard-major rows into token order, the reduce-scatter g-bar that sums t fp32 partials
// and writes shard-major rows, and dropout + residual add with a counter-hash mask; their
// backward (LayerNorm backward, dropout backward fused with the gather, fixed-order column
// and partial sums); RMSNorm ("Megatron 训练" notes, section "RMSNorm") through the LayerNorm
// kernels; and the attention block's two small helpers (softmax statistics combine, per-head
// row dot product of dO and O). All shards live in one HBM buffer [t][b][s/t][h], so g and
// g-bar are row permutations (plus the t-way sum for g-bar). Kernels move 16-byte vectors,
// with the shard <-> token mapping computed once per row.
#include "device_common.cuh"
#include <type_traits>

namespace tpmlp {
namespace {

// Token row r = bi*s + j*sl + l  <->  shard-major row R = (j*b + bi)*sl + l.
__device__ __forceinline__ int64_t shard_row_to_token(int64_t R, int64_t b, int64_t s, int64_t sl) {
  const int64_t jb = R / sl;
  const int64_t l = R - jb * sl;
  const int64_t j = jb / b;
  const int64_t bi = jb - j * b;
  return bi * s + j * sl + l;
}

template <typename T>
struct Vec8;  // 8 elements of T

template <>
struct Vec8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = u; }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = unpack_bf16x2(w[i]);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
  __device__ __forceinline__ void from_float(const float (&f)[8]) {
    u = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                   pack_bf16x2(f[6], f[7]));
  }
};

template <>
struct Vec8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void store(float* p) const {
    reinterpret_cast<float4*>(p)[0] = a;
    reinterpret_cast<float4*>(p)[1] = b;
  }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  __device__ __forceinline__ void from_float(const float (&f)[8]) {
    a = make_float4(f[0], f[1], f[2], f[3]);
    b = make_float4(f[4], f[5], f[6], f[7]);
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ LayerNorm
// One 128-thread CTA per row; each thread keeps CH vectors of 8 elements of the row in
// registers, so the row is read from HBM once and 16 rows per SM are in flight. Statistics
// in fp32: the mean, then the biased variance of the deviations (two passes over registers),
// each reduced across the CTA through shared memory that alternates between rows.
constexpr int kLnThreads = 128;

template <typename T, int CH>
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(const T* __restrict__ x,
                                                               const float* __restrict__ gamma,
                                                               const float* __restrict__ beta, float eps,
                                                               T* __restrict__ y, int64_t rows, int h) {
  __shared__ float red[2][2][kLnThreads / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  const float inv_h = 1.0f / static_cast<float>(h);
  int parity = 0;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, parity ^= 1) {
    const T* xr = x + r * h;
    Vec8<T> buf[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int c = (tid + kLnThreads * i) * 8;
      if (c < h) buf[i].load(xr + c);
    }
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      if ((tid + kLnThreads * i) * 8 < h) {
        float f[8];
        buf[i].to_float(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += f[e];
      }
    }
    sum = warp_sum(sum);
    if (lane == 0) red[parity][0][w] = sum;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < kLnThreads / 32; ++k) tot += red[parity][0][k];
    const float mean = tot * inv_h;
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      if ((tid + kLnThreads * i) * 8 < h) {
        float f[8];
        buf[i].to_float(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dlt = f[e] - mean;
          sq = fmaf(dlt, dlt, sq);
        }
      }
    }
    sq = warp_sum(sq);
    if (lane == 0) red[parity][1][w] = sq;
    __syncthreads();
    float var = 0.f;
#pragma unroll
    for (int k = 0; k < kLnThreads / 32; ++k) var += red[parity][1][k];
    const float rstd = rsqrtf(var * inv_h + eps);
    T* yr = y + r * h;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int c = (tid + kLnThreads * i) * 8;
      if (c < h) {
        const float4 g0 = reinterpret_cast<const float4*>(gamma + c)[0], g1 = reinterpret_cast<const float4*>(gamma + c)[1];
        const float4 b0 = reinterpret_cast<const float4*>(beta + c)[0], b1 = reinterpret_cast<const float4*>(beta + c)[1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        float f[8], o[8];
        buf[i].to_float(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf((f[e] - mean) * rstd, g[e], bb[e]);
        Vec8<T> out;
        out.from_float(o);
        out.store(yr + c);
      }
    }
  }
}

// Any width: one CTA per row, three passes over the row (it stays in L1/L2).
template <typename T>
__global__ void __launch_bounds__(256) layernorm_generic_kernel(const T* __restrict__ x,
                                                                const float* __restrict__ gamma,
                                                                const float* __restrict__ beta, float eps,
                                                                T* __restrict__ y, int64_t rows, int64_t h) {
  __shared__ float red[8];
  __shared__ float stat;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* xr = x + r * h;
    float acc = 0.f;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x) acc += static_cast<float>(xr[c]);
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < (blockDim.x >> 5); ++w) s += red[w];
      stat = s / static_cast<float>(h);
    }
    __syncthreads();
    const float mean = stat;
    __syncthreads();
    acc = 0.f;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x) {
      const float dlt = static_cast<float>(xr[c]) - mean;
      acc = fmaf(dlt, dlt, acc);
    }
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < (blockDim.x >> 5); ++w) s += red[w];
      stat = rsqrtf(s / static_cast<float>(h) + eps);
    }
    __syncthreads();
    const float rstd = stat;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x)
      y[r * h + c] = static_cast<T>(fmaf((static_cast<float>(xr[c]) - mean) * rstd, gamma[c], beta[c]));
    __syncthreads();
  }
}

// ------------------------------------------------------------------ gather (g forward)
// Destination row r (token order) <- source shard-major row; rows are copied as 16-byte vectors.
// Each CTA moves kRowsPer rows per iteration and every thread issues all its loads (up to
// kRowsPer * V vectors) before its stores, so enough bytes are in flight to cover HBM latency.
template <int V, int kRowsPer>
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     int64_t rows, int64_t b, int64_t s, int64_t sl, int row_vecs) {
  for (int64_t R0 = static_cast<int64_t>(blockIdx.x) * kRowsPer; R0 < rows;
       R0 += static_cast<int64_t>(gridDim.x) * kRowsPer) {
    uint4 v[kRowsPer][V];
#pragma unroll
    for (int k = 0; k < kRowsPer; ++k) {
      const int64_t R = R0 + k;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int c = threadIdx.x + j * 256;
        if (R < rows && c < row_vecs) v[k][j] = src[R * row_vecs + c];
      }
    }
#pragma unroll
    for (int k = 0; k < kRowsPer; ++k) {
      const int64_t R = R0 + k;
      if (R >= rows) break;
      uint4* dr = dst + shard_row_to_token(R, b, s, sl) * row_vecs;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int c = threadIdx.x + j * 256;
        if (c < row_vecs) dr[c] = v[k][j];
      }
    }
  }
}

// Any row width: one row per CTA iteration.
__global__ void __launch_bounds__(256) gather_generic_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                             int64_t rows, int64_t b, int64_t s, int64_t sl,
                                                             int row_vecs) {
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t r = shard_row_to_token(R, b, s, sl);
    const uint4* sr = src + R * row_vecs;
    uint4* dr = dst + r * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) dr[c] = sr[c];
  }
}

// ------------------------------------------------------------------ reduce-scatter (g-bar forward)
// Shard-major output row R <- sum over i = 0..t-1 (in order) of partials[i][token row].
template <typename T>
__global__ void __launch_bounds__(256) reduce_scatter_kernel(const float* __restrict__ partials, T* __restrict__ out,
                                                             int64_t rows, int64_t b, int64_t s, int64_t sl, int h,
                                                             int t) {
  const int64_t plane = rows * static_cast<int64_t>(h);
  const int nvec = h >> 3;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t r = shard_row_to_token(R, b, s, sl);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int c = v * 8;
      float acc[8];
      Vec8<float> p;
      p.load(partials + r * h + c);
      p.to_float(acc);
      for (int i = 1; i < t; ++i) {
        float f[8];
        p.load(partials + i * plane + r * h + c);
        p.to_float(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
      Vec8<T> o;
      o.from_float(acc);
      o.store(out + R * h + c);
    }
  }
}

// ------------------------------------------------------------------ dropout + residual

// Rare path of the dropout kernels (a key carrying into the hash's high word, a threshold of
// 2^63 or more, or a tie with the threshold's high word): the vector of 8 elements at k0 redone
// from global memory with eight full hashes, overwriting what the shortcut stored. y == nullptr
// selects the dropout gradient (out = keep * x * scale) instead of out = x + keep * y * scale.
template <typename T>
__device__ __noinline__ uint32_t dropout_vector_full(const T* xp, const T* yp, T* op, uint64_t base,
                                                     uint64_t threshold, float scale) {
  const uint32_t bits = drop_bits8_full(base, threshold);
  Vec8<T> xv;
  xv.load(xp);
  float xf[8], yf[8] = {}, o[8];
  xv.to_float(xf);
  if (yp != nullptr) {
    Vec8<T> yv;
    yv.load(yp);
    yv.to_float(yf);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const bool dropped = (bits >> e) & 1u;
    o[e] = yp != nullptr ? (dropped ? xf[e] : fmaf(yf[e], scale, xf[e])) : (dropped ? 0.f : xf[e] * scale);
  }
  Vec8<T> ov;
  ov.from_float(o);
  ov.store(op);
  return bits;
}

// Resident CTAs per SM of the dropout kernels: 16 x 128 threads, at most 32 registers a thread
// for bf16 (rows move through the memory system by occupancy, not by registers).
template <typename T>
constexpr int dropout_min_blocks() { return sizeof(T) == 2 ? 16 : 8; }

// out = x + keep * y * scale for shard-major rows; element k of the logical token-order
// tensor is dropped iff splitmix64(seed ^ k) < threshold. One thread per vector of 8
// consecutive elements, one row per CTA (grid = rows, so the block scheduler balances the
// tail); each element is decided by the high word of the last product (DropHash8) and the
// rare cases redo the vector in full. 4 neighbouring lanes OR their bits into one 32-bit
// mask word. kLow3 = seed & 7.
template <typename T, int kLow3>
__global__ void __launch_bounds__(128, dropout_min_blocks<T>()) dropout_residual_kernel(
    const T* __restrict__ x, const T* __restrict__ y, T* __restrict__ out, uint32_t* __restrict__ mask_bits,
    uint64_t threshold, float scale, uint64_t seed, int64_t rows, int64_t b, int64_t s, int64_t sl, int h) {
  const int nvec = h >> 3;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t r = shard_row_to_token(R, b, s, sl);
    const uint64_t flat_row = static_cast<uint64_t>(r) * static_cast<uint64_t>(h);
    const T* xr = x + R * h;
    const T* yr = y + R * h;
    T* orow = out + R * h;
    for (int v0 = 0; v0 < nvec; v0 += blockDim.x) {  // uniform trip count across the CTA
      const int v = v0 + threadIdx.x;
      uint32_t bits = 0;
      if (v < nvec) {
        const uint64_t base = seed ^ (flat_row + static_cast<uint64_t>(v) * 8);  // (seed^k0)^e = seed^(k0+e)
        const DropHash8<kLow3> hs(base, threshold);
        bool redo = !hs.shortcut;
        if (hs.shortcut) {
          Vec8<T> xv, yv;
          xv.load(xr + v * 8);
          yv.load(yr + v * 8);
          float xf[8], yf[8], o[8];
          xv.to_float(xf);
          yv.to_float(yf);
#pragma unroll
          for (uint32_t e = 0; e < 8; ++e) {
            const uint32_t c = hs.high(e);
            const bool dropped = c < hs.thi;
            redo |= c == hs.thi;
            bits |= (dropped ? 1u : 0u) << e;
            o[e] = dropped ? xf[e] : fmaf(yf[e], scale, xf[e]);
          }
          Vec8<T> ov;
          ov.from_float(o);
          ov.store(orow + v * 8);
        }
        if (redo) bits = dropout_vector_full(xr + v * 8, yr + v * 8, orow + v * 8, base, threshold, scale);
      }
      if (mask_bits != nullptr) {
        bits <<= 8 * (threadIdx.x & 3);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
        if (v < nvec && (threadIdx.x & 3) == 0) mask_bits[(flat_row + static_cast<uint64_t>(v) * 8) >> 5] = bits;
      }
    }
  }
}

// ------------------------------------------------------------------ bulk-copy row pipeline
// The staged kernels below stream whole rows through a shared-memory ring: CTA c handles rows
// R_i = c + i * gridDim.x, and thread 0 keeps up to kRowStages of them in flight with
// cp.async.bulk copies that complete on one mbarrier per stage, while every thread computes on
// rows already staged. Loads therefore never stall the computing warps. Every wait is bounded;
// the CTA agrees on a timeout through __syncthreads_or, thread 0 waits (bounded) for its copies
// still in flight, and the kernel returns.
__device__ __forceinline__ int64_t rows_for_cta(int64_t rows) {
  return rows > blockIdx.x ? (rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
}

template <int STAGES>
__device__ __forceinline__ void drain_rows(uint64_t* full, int64_t from, int64_t to, unsigned int* status) {
  for (int64_t k = from; k < to; ++k) mbar_wait(&full[k % STAGES], (k / STAGES) & 1, status, 21);
}


// LayerNorm with rows staged through the shared-memory ring; one CTA per row at a time, each
// thread holding CH vectors of 8 elements in registers. The statistics take one pass: every
// thread sums d = x - x_0 and d^2 (x_0, the row's first element, is a shift that keeps the
// one-pass variance E[d^2] - E[d]^2 free of cancellation for rows with a large mean), the
// warps' partial sums go to per-warp shared-memory slots that every thread adds in a fixed
// order after a single barrier (deterministic). Slots alternate between rows.
// kRms: RMSNorm ("Megatron 训练" notes, section "RMSNorm": LayerNorm without the mean):
// no shift, no mean, rstd = 1 / sqrt(mean(x^2) + eps), y = x * rstd * gamma (beta unused).
template <typename T, int CH, int kRowThreads, int kRowStages, bool kAffineInRegs, bool kRms = false>
__global__ void __launch_bounds__(kRowThreads)
    layernorm_staged_kernel(const T* __restrict__ x, const float* __restrict__ gamma, const float* __restrict__ beta,
                            float eps, T* __restrict__ y, int64_t rows, int h, unsigned int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float2 red[2][kRowThreads / 32];
  const uint32_t row_bytes = static_cast<uint32_t>(h) * sizeof(T);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRowStages * row_bytes);
  const int64_t nloc = rows_for_cta(rows);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < kRowStages; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int64_t i) {
    const int64_t R = blockIdx.x + i * gridDim.x;
    const int st = static_cast<int>(i % kRowStages);
    mbar_arrive_expect_tx(&full[st], row_bytes);
    bulk_load(smem + st * row_bytes, x + R * h, row_bytes, &full[st]);
  };
  if (tid == 0)
    for (int64_t i = 0; i < nloc && i < kRowStages; ++i) issue(i);
  // A thread touches the same columns of every row, so gamma and beta can stay in registers.
  float greg[kAffineInRegs ? CH : 1][8], breg[kAffineInRegs ? CH : 1][8];
  if constexpr (kAffineInRegs) {
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (tid + c * kRowThreads) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        greg[c][e] = col < h ? gamma[col + e] : 0.f;
        breg[c][e] = (!kRms && col < h) ? beta[col + e] : 0.f;
      }
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  int64_t i = 0;
  bool aborted = false;
  for (; i < nloc; ++i) {
    const int st = static_cast<int>(i % kRowStages);
    const int p = static_cast<int>(i & 1);
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>((i / kRowStages) & 1), status, 22);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const T* xs = reinterpret_cast<const T*>(smem + st * row_bytes);
    const float shift = kRms ? 0.f : static_cast<float>(xs[0]);
    float f[CH][8];
    float sum = 0.f, sq = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int v = tid + c * kRowThreads;
      if (v * 8 < h) {
        Vec8<T> in;
        in.load(xs + v * 8);
        in.to_float(f[c]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = f[c][e] - shift;
          sum += d;
          sq = fmaf(d, d, sq);
        }
      }
    }
    sum = warp_sum(sum);
    sq = warp_sum(sq);
    if (lane == 0) red[p][w] = make_float2(sum, sq);
    __syncthreads();  // the row's partial sums are published, and every thread has read stage st
    if (tid == 0 && i + kRowStages < nloc) issue(i + kRowStages);
    float tsum = 0.f, tsq = 0.f;
#pragma unroll
    for (int k = 0; k < kRowThreads / 32; ++k) {
      const float2 ps = red[p][k];
      tsum += ps.x;
      tsq += ps.y;
    }
    const float md = kRms ? 0.f : tsum * inv_h;  // mean of x - shift
    const float var = kRms ? tsq * inv_h : fmaxf(tsq * inv_h - md * md, 0.f);  // RMS: mean square
    const float rstd = rsqrtf(var + eps);
    const float a0 = kRms ? 0.f : -(md + shift) * rstd;  // (x - mean) * rstd = x * rstd + a0
    const int64_t R = blockIdx.x + i * gridDim.x;
    T* yr = y + R * h;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int v = tid + c * kRowThreads;
      if (v * 8 < h) {
        const int col = v * 8;
        float o[8];
        if constexpr (kAffineInRegs) {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = fmaf(fmaf(f[c][e], rstd, a0), greg[c][e], breg[c][e]);
        } else {
          const float4 g0 = reinterpret_cast<const float4*>(gamma + col)[0], g1 = reinterpret_cast<const float4*>(gamma + col)[1];
          float4 b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
          if constexpr (!kRms) {
            b0 = reinterpret_cast<const float4*>(beta + col)[0];
            b1 = reinterpret_cast<const float4*>(beta + col)[1];
          }
          const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = fmaf(fmaf(f[c][e], rstd, a0), g[e], bb[e]);
        }
        Vec8<T> ov;
        ov.from_float(o);
        ov.store(yr + col);
      }
    }
  }
  if (aborted && tid == 0) drain_rows<kRowStages>(full, i, i + kRowStages < nloc ? i + kRowStages : nloc, status);
}

// LayerNorm, one warp per row with no CTA-wide barriers: each warp streams its own rows
// (R = global warp index + i * total warps) through a private shared-memory ring filled by
// bulk copies, and reads each staged row three times (sum, squared deviations, output).
template <typename T, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
    layernorm_warp_staged_kernel(const T* __restrict__ x, const float* __restrict__ gamma,
                                 const float* __restrict__ beta, float eps, T* __restrict__ y, int64_t rows, int h,
                                 unsigned int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t row_bytes = static_cast<uint32_t>(h) * sizeof(T);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + static_cast<size_t>(warp) * STAGES * row_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(WARPS) * STAGES * row_bytes) + warp * STAGES;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * WARPS;
  const int64_t nloc = rows > gw ? (rows - 1 - gw) / nw + 1 : 0;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int64_t i) {
    const int st = static_cast<int>(i % STAGES);
    mbar_arrive_expect_tx(&full[st], row_bytes);
    bulk_load(ring + st * row_bytes, x + (gw + i * nw) * h, row_bytes, &full[st]);
  };
  if (lane == 0)
    for (int64_t i = 0; i < nloc && i < STAGES; ++i) issue(i);
  __syncwarp();
  const int nvec = h >> 3;
  const float inv_h = 1.0f / static_cast<float>(h);
  int64_t i = 0;
  bool aborted = false;
  for (; i < nloc; ++i) {
    const int st = static_cast<int>(i % STAGES);
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>((i / STAGES) & 1), status, 23);
    if (__any_sync(0xffffffffu, !ok)) {
      aborted = true;
      break;
    }
    const T* xs = reinterpret_cast<const T*>(ring + st * row_bytes);
    float sum = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      Vec8<T> in;
      in.load(xs + v * 8);
      float f[8];
      in.to_float(f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += f[e];
    }
    const float mean = warp_sum(sum) * inv_h;
    float sq = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      Vec8<T> in;
      in.load(xs + v * 8);
      float f[8];
      in.to_float(f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float dlt = f[e] - mean;
        sq = fmaf(dlt, dlt, sq);
      }
    }
    const float rstd = rsqrtf(warp_sum(sq) * inv_h + eps);
    T* yr = y + (gw + i * nw) * h;
    for (int v = lane; v < nvec; v += 32) {
      const int col = v * 8;
      Vec8<T> in;
      in.load(xs + col);
      float f[8], o[8];
      in.to_float(f);
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma + col));
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma + col) + 1);
      const float4 b0 = __ldg(reinterpret_cast<const float4*>(beta + col));
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(beta + col) + 1);
      const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = fmaf((f[e] - mean) * rstd, g[e], bb[e]);
      Vec8<T> out;
      out.from_float(o);
      out.store(yr + col);
    }
    __syncwarp();  // every lane has read stage st
    if (lane == 0 && i + STAGES < nloc) issue(i + STAGES);
  }
  if (aborted && lane == 0) drain_rows<STAGES>(full, i, i + STAGES < nloc ? i + STAGES : nloc, status);
}

// Dynamic shared memory of a staged kernel: the row ring plus one mbarrier per stage.
size_t staged_smem(size_t stage_bytes, int stages) { return stages * stage_bytes + stages * sizeof(uint64_t); }

constexpr int kLnStagedThreads = 128, kLnStages = 6;
constexpr bool kLnAffineInRegs = true;  // gamma, beta read once per CTA

constexpr size_t kStagedSmemMax = 100 * 1024;  // at least two CTAs per SM

// ------------------------------------------------------------------ SP backward kernels
// Inverse of shard_row_to_token: token row r = bi*s + j*sl + l -> shard-major row (j*b + bi)*sl + l.
__device__ __forceinline__ int64_t token_to_shard_row(int64_t r, int64_t b, int64_t s, int64_t sl) {
  const int64_t bi = r / s;
  const int64_t si = r - bi * s;
  const int64_t j = si / sl;
  return (j * b + bi) * sl + (si - j * sl);
}

// Dropout backward fused with g-bar's backward (all-gather): token row r of the result is
// dout[shard row of r] * keep / (1 - p), with the mask recomputed from the hash; one thread
// per vector of 8 elements, one token row per CTA, as dropout_residual_kernel. kLow3 = seed & 7.
template <typename T, int kLow3>
__global__ void __launch_bounds__(128, dropout_min_blocks<T>()) dropout_grad_gather_kernel(
    const T* __restrict__ dout, T* __restrict__ dtok, uint64_t threshold, float scale, uint64_t seed, int64_t rows,
    int64_t b, int64_t s, int64_t sl, int h) {
  const int nvec = h >> 3;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* src = dout + token_to_shard_row(r, b, s, sl) * h;
    T* dst = dtok + r * h;
    const uint64_t flat_row = static_cast<uint64_t>(r) * static_cast<uint64_t>(h);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const uint64_t base = seed ^ (flat_row + static_cast<uint64_t>(v) * 8);
      const DropHash8<kLow3> hs(base, threshold);
      bool redo = !hs.shortcut;
      if (hs.shortcut) {
        Vec8<T> gv;
        gv.load(src + v * 8);
        float gf[8], o[8];
        gv.to_float(gf);
#pragma unroll
        for (uint32_t e = 0; e < 8; ++e) {
          const uint32_t c = hs.high(e);
          redo |= c == hs.thi;
          o[e] = c < hs.thi ? 0.f : gf[e] * scale;
        }
        Vec8<T> ov;
        ov.from_float(o);
        ov.store(dst + v * 8);
      }
      if (redo) dropout_vector_full<T>(src + v * 8, nullptr, dst + v * 8, base, threshold, scale);
    }
  }
}

// LayerNorm backward plus the residual, one CTA per row (persistent over rows):
//   dx = dout + rstd * (g - mean(g) - x_hat * mean(g * x_hat)),  g = dxn * gamma,
// with the row statistics recomputed from x in one shifted pass and all four row sums
// (sum d, sum d^2, sum g, sum g*d with d = x - x_0) reduced together. Each thread owns CH
// vectors of columns and accumulates dgamma (dxn * x_hat) and dbeta (dxn) for them over its
// CTA's rows in its own slots of a shared-memory array laid out [2][CH][8][threads] (no two
// threads share a slot, so no atomics, and a warp's accesses hit 32 consecutive words, so no
// bank conflicts); the CTA writes them to partials[blockIdx][2][h] for a fixed-order sum.
constexpr int kLnBwdThreads = 128;

// kRms: RMSNorm's backward, dx = [dout +] rstd * (g - x_hat * mean(g * x_hat)) with
// x_hat = x * rstd (no shift, no mean, no mean(g) term). dout may be null (no residual).
template <typename T, int CH, bool kRms = false>
__global__ void __launch_bounds__(kLnBwdThreads, 4)
    layernorm_backward_kernel(const T* __restrict__ x, const T* __restrict__ dxn, const T* __restrict__ dout,
                              const float* __restrict__ gamma, float eps, T* __restrict__ dx,
                              float* __restrict__ partials, int64_t rows, int h) {
  __shared__ float4 red[2][kLnBwdThreads / 32];
  extern __shared__ float acc[];  // [2][CH][8][kLnBwdThreads]: dgamma then dbeta partial sums
  constexpr int kHalf = CH * 8 * kLnBwdThreads;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  float gam[CH][8];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int col = (tid + c * kLnBwdThreads) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      gam[c][e] = col < h ? gamma[col + e] : 0.f;
      acc[(c * 8 + e) * kLnBwdThreads + tid] = 0.f;
      acc[kHalf + (c * 8 + e) * kLnBwdThreads + tid] = 0.f;
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  int p = 0;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x, p ^= 1) {
    const T* xr = x + R * h;
    const T* dr = dxn + R * h;
    const T* gr = dout ? dout + R * h : nullptr;
    const float shift = kRms ? 0.f : static_cast<float>(xr[0]);
    float f[CH][8], dn[CH][8];
    Vec8<T> gv[CH];  // dout, loaded with x and dxn so that all of the row's reads are in flight at once
    float s_d = 0.f, s_dd = 0.f, s_g = 0.f, s_gd = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (tid + c * kLnBwdThreads) * 8;
      if (col < h) {
        Vec8<T> xv, dv;
        xv.load(xr + col);
        dv.load(dr + col);
        if (gr) gv[c].load(gr + col);
        xv.to_float(f[c]);
        dv.to_float(dn[c]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = f[c][e] - shift;
          const float g = dn[c][e] * gam[c][e];
          if constexpr (!kRms) {
            s_d += d;
            s_g += g;
          }
          s_dd = fmaf(d, d, s_dd);
          s_gd = fmaf(g, d, s_gd);
        }
      }
    }
    if constexpr (!kRms) {
      s_d = warp_sum(s_d);
      s_g = warp_sum(s_g);
    }
    s_dd = warp_sum(s_dd);
    s_gd = warp_sum(s_gd);
    if (lane == 0) red[p][w] = make_float4(s_d, s_dd, s_g, s_gd);
    __syncthreads();
    float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kLnBwdThreads / 32; ++k) {
      const float4 v = red[p][k];
      t4.x += v.x;
      t4.y += v.y;
      t4.z += v.z;
      t4.w += v.w;
    }
    const float md = kRms ? 0.f : t4.x * inv_h;
    const float rstd = rsqrtf((kRms ? t4.y * inv_h : fmaxf(t4.y * inv_h - md * md, 0.f)) + eps);
    const float mean_g = kRms ? 0.f : t4.z * inv_h;
    const float mean_gxh = rstd * (t4.w * inv_h - md * mean_g);  // mean(g * x_hat)
    T* outr = dx + R * h;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (tid + c * kLnBwdThreads) * 8;
      if (col < h) {
        float go[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, o[8];
        if (gr) gv[c].to_float(go);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = (f[c][e] - shift - md) * rstd;
          const float g = dn[c][e] * gam[c][e];
          o[e] = go[e] + rstd * (g - mean_g - xh * mean_gxh);
          const int slot = (c * 8 + e) * kLnBwdThreads + tid;
          acc[slot] = fmaf(dn[c][e], xh, acc[slot]);
          acc[kHalf + slot] += dn[c][e];
        }
        Vec8<T> ov;
        ov.from_float(o);
        ov.store(outr + col);
      }
    }
  }
  float* pg = partials + static_cast<int64_t>(blockIdx.x) * 2 * h;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int col = (tid + c * kLnBwdThreads) * 8;
    if (col < h) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pg[col + e] = acc[(c * 8 + e) * kLnBwdThreads + tid];
        pg[h + col + e] = acc[kHalf + (c * 8 + e) * kLnBwdThreads + tid];
      }
    }
  }
}

// The same backward (LayerNorm, or RMSNorm with kRms) with the row streamed through the
// bulk-copy ring: thread 0 keeps `stages` rows of x, dxn (and dout when given) in flight, so
// loads never wait behind the reductions. 256 threads, CH vectors of 8 columns per thread;
// dgamma / dbeta accumulate in registers and go to partials[blockIdx][2][h] at the end.
// Needs 16-byte aligned row starts (bulk copies).
constexpr int kLnBwdStagedThreads = 256;

template <typename T, int CH, bool kRms>
__global__ void __launch_bounds__(kLnBwdStagedThreads)
    norm_backward_staged_kernel(const T* __restrict__ x, const T* __restrict__ dxn, const T* __restrict__ dout,
                                const float* __restrict__ gamma, float eps, T* __restrict__ dx,
                                float* __restrict__ partials, int64_t rows, int h, int stages,
                                unsigned int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float4 red[2][kLnBwdStagedThreads / 32];
  const uint32_t row_bytes = static_cast<uint32_t>(h) * sizeof(T);
  const uint32_t stage_bytes = (dout ? 3u : 2u) * row_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(stages) * stage_bytes);
  const int64_t nloc = rows_for_cta(rows);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int64_t i) {
    const int64_t R = blockIdx.x + i * gridDim.x;
    const int st = static_cast<int>(i % stages);
    uint8_t* dst = smem + static_cast<size_t>(st) * stage_bytes;
    mbar_arrive_expect_tx(&full[st], stage_bytes);
    bulk_load(dst, x + R * h, row_bytes, &full[st]);
    bulk_load(dst + row_bytes, dxn + R * h, row_bytes, &full[st]);
    if (dout) bulk_load(dst + 2 * row_bytes, dout + R * h, row_bytes, &full[st]);
  };
  if (tid == 0)
    for (int64_t i = 0; i < nloc && i < stages; ++i) issue(i);
  float gam[CH][8], accg[CH][8], accb[kRms ? 1 : CH][8];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int col = (tid + c * kLnBwdStagedThreads) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      gam[c][e] = col < h ? gamma[col + e] : 0.f;
      accg[c][e] = 0.f;
      if constexpr (!kRms) accb[c][e] = 0.f;
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  int64_t i = 0;
  bool aborted = false;
  for (; i < nloc; ++i) {
    const int st = static_cast<int>(i % stages);
    const int p = static_cast<int>(i & 1);
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>((i / stages) & 1), status, 23);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const T* xs = reinterpret_cast<const T*>(smem + static_cast<size_t>(st) * stage_bytes);
    const T* ds = reinterpret_cast<const T*>(smem + static_cast<size_t>(st) * stage_bytes + row_bytes);
    const T* gs = reinterpret_cast<const T*>(smem + static_cast<size_t>(st) * stage_bytes + 2 * row_bytes);
    const float shift = kRms ? 0.f : static_cast<float>(xs[0]);
    float f[CH][8], dn[CH][8], go[CH][8];
    float s_d = 0.f, s_dd = 0.f, s_g = 0.f, s_gd = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (tid + c * kLnBwdStagedThreads) * 8;
      if (col < h) {
        Vec8<T> xv, dv;
        xv.load(xs + col);
        dv.load(ds + col);
        xv.to_float(f[c]);
        dv.to_float(dn[c]);
        if (dout) {
          Vec8<T> gv;
          gv.load(gs + col);
          gv.to_float(go[c]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) go[c][e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = f[c][e] - shift;
          const float g = dn[c][e] * gam[c][e];
          if constexpr (!kRms) {
            s_d += d;
            s_g += g;
          }
          s_dd = fmaf(d, d, s_dd);
          s_gd = fmaf(g, d, s_gd);
        }
      }
    }
    if constexpr (!kRms) {
      s_d = warp_sum(s_d);
      s_g = warp_sum(s_g);
    }
    s_dd = warp_sum(s_dd);
    s_gd = warp_sum(s_gd);
    if (lane == 0) red[p][w] = make_float4(s_d, s_dd, s_g, s_gd);
    __syncthreads();  // the row's sums are published, and every thread has read stage st
    if (tid == 0 && i + stages < nloc) issue(i + stages);
    float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kLnBwdStagedThreads / 32; ++k) {
      const float4 v = red[p][k];
      t4.x += v.x;
      t4.y += v.y;
      t4.z += v.z;
      t4.w += v.w;
    }
    const float md = kRms ? 0.f : t4.x * inv_h;
    const float rstd = rsqrtf((kRms ? t4.y * inv_h : fmaxf(t4.y * inv_h - md * md, 0.f)) + eps);
    const float mean_g = kRms ? 0.f : t4.z * inv_h;
    const float mean_gxh = rstd * (t4.w * inv_h - md * mean_g);  // mean(g * x_hat)
    const int64_t R = blockIdx.x + i * gridDim.x;
    T* outr = dx + R * h;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int col = (tid + c * kLnBwdStagedThreads) * 8;
      if (col < h) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = (f[c][e] - shift - md) * rstd;
          const float g = dn[c][e] * gam[c][e];
          o[e] = go[c][e] + rstd * (g - mean_g - xh * mean_gxh);
          accg[c][e] = fmaf(dn[c][e], xh, accg[c][e]);
          if constexpr (!kRms) accb[c][e] += dn[c][e];
        }
        Vec8<T> ov;
        ov.from_float(o);
        ov.store(outr + col);
      }
    }
  }
  if (aborted && tid == 0)
    for (int64_t k = i; k < nloc && k < i + stages; ++k) mbar_wait(&full[k % stages], (k / stages) & 1, status, 21);
  float* pg = partials + static_cast<int64_t>(blockIdx.x) * 2 * h;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int col = (tid + c * kLnBwdStagedThreads) * 8;
    if (col < h) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pg[col + e] = accg[c][e];
        pg[h + col + e] = kRms ? 0.f : accb[kRms ? 0 : c][e];
      }
    }
  }
}

// dgamma[c] = sum over CTAs of partials[k][0][c], dbeta likewise. A CTA takes 32 of the 2h
// columns; thread (g, c) adds partials g, g+8, g+16, ... of its column, and the 8 group sums are
// then added in group order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(256) sum_partials_kernel(const float* __restrict__ partials, int nparts, int h,
                                                           float* __restrict__ dgamma, float* __restrict__ dbeta) {
  __shared__ float grp[8][32];
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float acc = 0.f;
  if (c < 2 * h)
    for (int k = g; k < nparts; k += 8) acc += partials[static_cast<int64_t>(k) * 2 * h + c];
  grp[g][lane] = acc;
  __syncthreads();
  if (g == 0 && c < 2 * h) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += grp[k][lane];
    if (c < h) dgamma[c] = t;
    else if (dbeta) dbeta[c - h] = t;
  }
}

// ------------------------------------------------------------------ column sums (bias gradients)
// Pass 1: CTA (x, y) sums rows [y*kColSumRows, (y+1)*kColSumRows) of 8 columns per thread.
template <typename T>
__global__ void __launch_bounds__(256) colsum_partial_kernel(const T* __restrict__ M, int64_t rows, int cols,
                                                             float* __restrict__ partials) {
  const int64_t cg = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int c0 = static_cast<int>(cg * 8);
  if (c0 >= cols) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kColSumRows;
  const int64_t r1 = r0 + kColSumRows < rows ? r0 + kColSumRows : rows;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c0 + 8 <= cols && (cols % 8) == 0) {
#pragma unroll 4
    for (int64_t r = r0; r < r1; ++r) {
      Vec8<T> v;
      v.load(M + r * cols + c0);
      float f[8];
      v.to_float(f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += f[e];
    }
  } else {
    for (int64_t r = r0; r < r1; ++r)
      for (int e = 0; e < 8 && c0 + e < cols; ++e) acc[e] += static_cast<float>(M[r * cols + c0 + e]);
  }
  float* pr = partials + static_cast<int64_t>(blockIdx.y) * cols;
  for (int e = 0; e < 8 && c0 + e < cols; ++e) pr[c0 + e] = acc[e];
}

// Pass 2: out[c] = sum of partials[k][c] over chunks k in order.
__global__ void __launch_bounds__(256) colsum_final_kernel(const float* __restrict__ partials, int chunks, int cols,
                                                           float* __restrict__ out) {
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int k = 0; k < chunks; ++k) acc += partials[static_cast<int64_t>(k) * cols + c];
    out[c] = acc;
  }
}

// ------------------------------------------------------------------ attention softmax (fused form)
// Row r's partial statistics (m_j, l_j) from the scores GEMM's kEpiRowStats epilogue (base 2:
// m_j = max of the scaled scores times log2(e), l_j = sum of 2^(y - m_j)) become M = max_j m_j
// and 1/L with L = sum_j l_j * 2^(m_j - M); one warp per row, lanes over j.
__global__ void __launch_bounds__(256) softmax_combine_kernel(const float2* __restrict__ stats, int nparts,
                                                              float2* __restrict__ rowstats, int64_t rows) {
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;  // uniform across the warp
  const float2* st = stats + r * nparts;
  float2 v[2];
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int j = lane + 32 * k;
    v[k] = j < nparts ? st[j] : make_float2(-INFINITY, 0.f);
    M = fmaxf(M, v[k].x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) L += v[k].y > 0.f ? v[k].y * ex2_approx(v[k].x - M) : 0.f;
  L = warp_sum(L);
  if (lane == 0) rowstats[r] = make_float2(M, 1.0f / L);
}

// D[(bi*heads + j)*s + si] = sum over head j's dh columns of dO * O in token row bi*s + si
// (= rowsum(P * dP) for that query row). One warp per token row; the lanes read a head's dh/8
// 16-byte vectors of dO and O (coalesced), several heads at once when dh/8 divides 32, and the
// products are summed across the lanes of each head.
__global__ void __launch_bounds__(256) row_dot_kernel(const __nv_bfloat16* __restrict__ dO,
                                                      const __nv_bfloat16* __restrict__ O, float* __restrict__ D,
                                                      int64_t b, int64_t s, int64_t h, int heads) {
  const int64_t tok = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (tok >= b * s) return;  // uniform across the warp
  const int64_t dh = h / heads;
  const int vh = static_cast<int>(dh / 8);
  const int64_t bi = tok / s, si = tok - bi * s;
  const __nv_bfloat16* a = dO + tok * h;
  const __nv_bfloat16* c = O + tok * h;
  if (vh <= 32 && (32 % vh) == 0) {
    // 32 / vh heads at a time: lane l takes vector l % vh of head j0 + l / vh; segments of vh
    // lanes are summed by xor shuffles that stay inside the segment.
    const int hpw = 32 / vh, seg = lane / vh, v = lane % vh;
    for (int j0 = 0; j0 < heads; j0 += hpw) {
      const int j = j0 + seg;
      float acc = 0.f;
      if (j < heads) {
        Vec8<__nv_bfloat16> va, vc;
        va.load(a + j * dh + v * 8);
        vc.load(c + j * dh + v * 8);
        float fa[8], fc[8];
        va.to_float(fa);
        vc.to_float(fc);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = fmaf(fa[k], fc[k], acc);
      }
      for (int o = vh / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (v == 0 && j < heads) D[(bi * heads + j) * s + si] = acc;
    }
    return;
  }
  for (int j = 0; j < heads; ++j) {
    float acc = 0.f;
    for (int v = lane; v < vh; v += 32) {
      Vec8<__nv_bfloat16> va, vc;
      va.load(a + j * dh + v * 8);
      vc.load(c + j * dh + v * 8);
      float fa[8], fc[8];
      va.to_float(fa);
      vc.to_float(fc);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(fa[k], fc[k], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) D[(bi * heads + j) * s + si] = acc;
  }
}

int rows_grid(int64_t rows, int num_sms, int per_sm) {
  const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
  return static_cast<int>(rows < cap ? (rows > 0 ? rows : 1) : cap);
}

}  // namespace

cudaError_t launch_layernorm(const void* x, const float* gamma, const float* beta, float eps, void* y, int64_t rows,
                             int64_t h, bool bf16, cudaStream_t stream, int num_sms, unsigned int* status, bool rms) {
  if (rows <= 0) return cudaSuccess;
  const size_t elt = bf16 ? 2 : 4;
  const size_t ln_smem = staged_smem(static_cast<size_t>(h) * elt, kLnStages);
  const bool staged = h % 8 == 0 && h <= kLnStagedThreads * 8 * 8 && ln_smem <= kStagedSmemMax;
  if (rms && !staged) return cudaErrorNotSupported;  // RMSNorm runs on the staged kernel only
  if (staged) {
    const int by_smem = static_cast<int>((220 * 1024) / ln_smem);
    const int by_threads = 2048 / kLnStagedThreads;
    const int per_sm = by_smem < by_threads ? (by_smem > 0 ? by_smem : 1) : by_threads;
    const int grid = rows_grid(rows, num_sms, per_sm);
    const int ch = static_cast<int>((h / 8 + kLnStagedThreads - 1) / kLnStagedThreads);
#define TPMLP_LN_STAGED(TYPE, CHN)                                                                              \
  do {                                                                                                          \
    auto k = rms ? layernorm_staged_kernel<TYPE, CHN, kLnStagedThreads, kLnStages, kLnAffineInRegs, true>       \
                 : layernorm_staged_kernel<TYPE, CHN, kLnStagedThreads, kLnStages, kLnAffineInRegs, false>;     \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ln_smem);         \
    if (e != cudaSuccess) return e;                                                                             \
    k<<<grid, kLnStagedThreads, ln_smem, stream>>>(static_cast<const TYPE*>(x), gamma, beta, eps,               \
                                                   static_cast<TYPE*>(y), rows, (int)h, status);                \
  } while (0)
    if (bf16) {
      if (ch <= 1) TPMLP_LN_STAGED(__nv_bfloat16, 1);
      else if (ch <= 2) TPMLP_LN_STAGED(__nv_bfloat16, 2);
      else if (ch <= 4) TPMLP_LN_STAGED(__nv_bfloat16, 4);
      else TPMLP_LN_STAGED(__nv_bfloat16, 8);
    } else {
      if (ch <= 1) TPMLP_LN_STAGED(float, 1);
      else if (ch <= 2) TPMLP_LN_STAGED(float, 2);
      else if (ch <= 4) TPMLP_LN_STAGED(float, 4);
      else TPMLP_LN_STAGED(float, 8);
    }
#undef TPMLP_LN_STAGED
  } else if ((h % 8 == 0) && (h <= kLnThreads * 8 * 8)) {
    const int grid = rows_grid(rows, num_sms, 16);
    const int ch = static_cast<int>((h / 8 + kLnThreads - 1) / kLnThreads);
    if (bf16) {
      auto xp = static_cast<const __nv_bfloat16*>(x);
      auto yp = static_cast<__nv_bfloat16*>(y);
      if (ch <= 1) layernorm_kernel<__nv_bfloat16, 1><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else if (ch <= 2) layernorm_kernel<__nv_bfloat16, 2><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else if (ch <= 4) layernorm_kernel<__nv_bfloat16, 4><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else layernorm_kernel<__nv_bfloat16, 8><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
    } else {
      auto xp = static_cast<const float*>(x);
      auto yp = static_cast<float*>(y);
      if (ch <= 1) layernorm_kernel<float, 1><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else if (ch <= 2) layernorm_kernel<float, 2><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else if (ch <= 4) layernorm_kernel<float, 4><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else layernorm_kernel<float, 8><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
    }
  } else {
    const int grid = rows_grid(rows, num_sms, 8);
    if (bf16)
      layernorm_generic_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), gamma, beta, eps, static_cast<__nv_bfloat16*>(y), rows, h);
    else
      layernorm_generic_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), gamma, beta, eps,
                                                                 static_cast<float*>(y), rows, h);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x_shards, void* x_full, int64_t b, int64_t s, int64_t h, int t, bool bf16,
                          cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  const int64_t row_bytes = h * (bf16 ? 2 : 4);
  if (row_bytes % 16 != 0) return cudaErrorInvalidValue;
  const int row_vecs = static_cast<int>(row_bytes / 16);
  const auto* src = static_cast<const uint4*>(x_shards);
  auto* dst = static_cast<uint4*>(x_full);
  if (row_vecs <= 256) {
    gather_kernel<1, 4><<<rows_grid((rows + 3) / 4, num_sms, 8), 256, 0, stream>>>(src, dst, rows, b, s, s / t, row_vecs);
  } else if (row_vecs <= 512) {
    // one row per CTA up to 64 CTAs per SM: the block scheduler balances the tail
    gather_kernel<2, 1><<<rows_grid(rows, num_sms, 64), 256, 0, stream>>>(src, dst, rows, b, s, s / t, row_vecs);
  } else if (row_vecs <= 1024) {
    gather_kernel<4, 1><<<rows_grid(rows, num_sms, 8), 256, 0, stream>>>(src, dst, rows, b, s, s / t, row_vecs);
  } else {
    gather_generic_kernel<<<rows_grid(rows, num_sms, 8), 256, 0, stream>>>(src, dst, rows, b, s, s / t, row_vecs);
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_scatter(const float* partials, void* out_shards, int64_t b, int64_t s, int64_t h, int t,
                                  bool bf16, cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0) return cudaErrorInvalidValue;
  const int grid = rows_grid(rows, num_sms, 8);
  if (bf16)
    reduce_scatter_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(partials, static_cast<__nv_bfloat16*>(out_shards),
                                                                    rows, b, s, s / t, static_cast<int>(h), t);
  else
    reduce_scatter_kernel<float><<<grid, 256, 0, stream>>>(partials, static_cast<float*>(out_shards), rows, b, s,
                                                            s / t, static_cast<int>(h), t);
  return cudaGetLastError();
}

// Calls launch(std::integral_constant<int, seed & 7>{}): the dropout kernels take the seed's low
// three bits as a template argument.
template <class L>
cudaError_t with_seed_low3(uint64_t seed, L&& launch) {
  switch (static_cast<int>(seed & 7)) {
    case 0: launch(std::integral_constant<int, 0>{}); break;
    case 1: launch(std::integral_constant<int, 1>{}); break;
    case 2: launch(std::integral_constant<int, 2>{}); break;
    case 3: launch(std::integral_constant<int, 3>{}); break;
    case 4: launch(std::integral_constant<int, 4>{}); break;
    case 5: launch(std::integral_constant<int, 5>{}); break;
    case 6: launch(std::integral_constant<int, 6>{}); break;
    default: launch(std::integral_constant<int, 7>{}); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dropout_residual(const void* x_shards, const void* y_shards, void* out_shards,
                                    uint32_t* mask_bits, uint64_t threshold, float scale, uint64_t seed, int64_t b,
                                    int64_t s, int64_t h, int t, bool bf16, cudaStream_t stream, int num_sms,
                                    unsigned int* status) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0 || (mask_bits && h % 32 != 0)) return cudaErrorInvalidValue;
  const int grid = rows_grid(rows, num_sms, 64);  // one row per CTA up to 64 CTAs per SM
  return with_seed_low3(seed, [&](auto low3) {
    constexpr int kLow3 = decltype(low3)::value;
    if (bf16)
      dropout_residual_kernel<__nv_bfloat16, kLow3><<<grid, 128, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x_shards), static_cast<const __nv_bfloat16*>(y_shards),
          static_cast<__nv_bfloat16*>(out_shards), mask_bits, threshold, scale, seed, rows, b, s, s / t,
          static_cast<int>(h));
    else
      dropout_residual_kernel<float, kLow3><<<grid, 128, 0, stream>>>(
          static_cast<const float*>(x_shards), static_cast<const float*>(y_shards), static_cast<float*>(out_shards),
          mask_bits, threshold, scale, seed, rows, b, s, s / t, static_cast<int>(h));
  });
}

cudaError_t launch_dropout_grad_gather(const void* dout_shards, void* dtok, uint64_t threshold, float scale,
                                       uint64_t seed, int64_t b, int64_t s, int64_t h, int t, bool bf16,
                                       cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0) return cudaErrorInvalidValue;
  const int grid = rows_grid(rows, num_sms, 64);  // one row per CTA up to 64 CTAs per SM
  return with_seed_low3(seed, [&](auto low3) {
    constexpr int kLow3 = decltype(low3)::value;
    if (bf16)
      dropout_grad_gather_kernel<__nv_bfloat16, kLow3><<<grid, 128, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(dout_shards), static_cast<__nv_bfloat16*>(dtok), threshold, scale, seed,
          rows, b, s, s / t, static_cast<int>(h));
    else
      dropout_grad_gather_kernel<float, kLow3><<<grid, 128, 0, stream>>>(
          static_cast<const float*>(dout_shards), static_cast<float*>(dtok), threshold, scale, seed, rows, b, s,
          s / t, static_cast<int>(h));
  });
}

cudaError_t launch_column_sums(const void* M, int64_t rows, int64_t cols, bool bf16, float* partials, float* out,
                               cudaStream_t stream) {
  if (cols <= 0) return cudaSuccess;
  if (rows <= 0) return cudaMemsetAsync(out, 0, sizeof(float) * cols, stream);
  const int64_t chunks = (rows + kColSumRows - 1) / kColSumRows;
  if (chunks > 65535 || cols > INT32_MAX) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>((cols / 8 + 1 + 255) / 256), static_cast<unsigned>(chunks));
  if (bf16)
    colsum_partial_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(M), rows,
                                                                    static_cast<int>(cols), partials);
  else
    colsum_partial_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(M), rows,
                                                            static_cast<int>(cols), partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  colsum_final_kernel<<<static_cast<unsigned>((cols + 255) / 256), 256, 0, stream>>>(
      partials, static_cast<int>(chunks), static_cast<int>(cols), out);
  return cudaGetLastError();
}

// One resident wave: as many CTAs as fit on the SMs at once (by registers and shared memory),
// so no CTA waits for another to finish; at most kLnBwdMaxCtas (the partials' capacity).
template <typename KERN>
int layernorm_backward_grid(KERN kernel, size_t smem, int64_t rows, int num_sms) {
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLnBwdThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int g = rows_grid(rows, num_sms, per_sm);
  return g < kLnBwdMaxCtas ? g : kLnBwdMaxCtas;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_layernorm_backward(const void* x, const void* dxn, const void* dout, const float* gamma, float eps,
                                      void* dx, float* partials, float* dgamma, float* dbeta, int64_t rows, int64_t h,
                                      bool bf16, cudaStream_t stream, int num_sms, bool rms, unsigned int* status) {
  if (rows <= 0) return cudaSuccess;
  const size_t elt = bf16 ? 2 : 4;
  const size_t stage_bytes = (dout ? 3 : 2) * static_cast<size_t>(h) * elt;
  const bool staged = h % 8 == 0 && h <= kLnBwdStagedThreads * 8 * 2 && aligned16(x) && aligned16(dxn) &&
                      (!dout || aligned16(dout)) && 2 * stage_bytes + 16 <= kStagedSmemMax;
  if (staged) {
    int stages = static_cast<int>(kStagedSmemMax / (stage_bytes + sizeof(uint64_t)));
    stages = stages > 4 ? 4 : stages;
    const size_t smem = staged_smem(stage_bytes, stages);
    const int ch = static_cast<int>((h / 8 + kLnBwdStagedThreads - 1) / kLnBwdStagedThreads);
    int grid = 0;
#define TPMLP_NBS(TYPE, CHN)                                                                                       \
  do {                                                                                                             \
    auto k = rms ? norm_backward_staged_kernel<TYPE, CHN, true> : norm_backward_staged_kernel<TYPE, CHN, false>;   \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);               \
    if (e != cudaSuccess) return e;                                                                                \
    int per_sm = 1;                                                                                                \
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kLnBwdStagedThreads, smem) != cudaSuccess ||     \
        per_sm < 1)                                                                                                \
      per_sm = 1;                                                                                                  \
    grid = rows_grid(rows, num_sms, per_sm);                                                                       \
    grid = grid < kLnBwdMaxCtas ? grid : kLnBwdMaxCtas;                                                            \
    k<<<grid, kLnBwdStagedThreads, smem, stream>>>(static_cast<const TYPE*>(x), static_cast<const TYPE*>(dxn),     \
                                                   static_cast<const TYPE*>(dout), gamma, eps, static_cast<TYPE*>(dx), \
                                                   partials, rows, static_cast<int>(h), stages, status);          \
  } while (0)
    if (bf16) {
      if (ch <= 1) TPMLP_NBS(__nv_bfloat16, 1);
      else TPMLP_NBS(__nv_bfloat16, 2);
    } else {
      if (ch <= 1) TPMLP_NBS(float, 1);
      else TPMLP_NBS(float, 2);
    }
#undef TPMLP_NBS
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int hb = static_cast<int>((2 * h + 31) / 32);
    sum_partials_kernel<<<hb, 256, 0, stream>>>(partials, grid, static_cast<int>(h), dgamma, dbeta);
    return cudaGetLastError();
  }
  if (h % 8 != 0 || h > kLnBwdThreads * 8 * 4) return cudaErrorInvalidValue;
  const int ch = static_cast<int>((h / 8 + kLnBwdThreads - 1) / kLnBwdThreads);
  const size_t acc_bytes = 2 * static_cast<size_t>(ch) * 8 * kLnBwdThreads * sizeof(float);  // <= 32 KiB
  int grid = 0;
#define TPMLP_LNB(TYPE, CHN)                                                                                     \
  do {                                                                                                           \
    auto k = rms ? layernorm_backward_kernel<TYPE, CHN, true> : layernorm_backward_kernel<TYPE, CHN, false>;    \
    grid = layernorm_backward_grid(k, acc_bytes, rows, num_sms);                                                 \
    k<<<grid, kLnBwdThreads, acc_bytes, stream>>>(static_cast<const TYPE*>(x), static_cast<const TYPE*>(dxn),    \
                                                  static_cast<const TYPE*>(dout), gamma, eps,                   \
                                                  static_cast<TYPE*>(dx), partials, rows, static_cast<int>(h)); \
  } while (0)
  if (bf16) {
    if (ch <= 1) TPMLP_LNB(__nv_bfloat16, 1);
    else if (ch <= 2) TPMLP_LNB(__nv_bfloat16, 2);
    else TPMLP_LNB(__nv_bfloat16, 4);
  } else {
    if (ch <= 1) TPMLP_LNB(float, 1);
    else if (ch <= 2) TPMLP_LNB(float, 2);
    else TPMLP_LNB(float, 4);
  }
#undef TPMLP_LNB
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int hb = static_cast<int>((2 * h + 31) / 32);
  sum_partials_kernel<<<hb, 256, 0, stream>>>(partials, grid, static_cast<int>(h), dgamma, dbeta);
  return cudaGetLastError();
}

cudaError_t launch_softmax_combine(const void* stats, int nparts, void* rowstats, int64_t rows, cudaStream_t stream,
                                   int num_sms) {
  (void)num_sms;
  if (rows <= 0) return cudaSuccess;
  if (nparts > 64) return cudaErrorInvalidValue;  // s <= 8192: at most 2 * 32 parts
  softmax_combine_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const float2*>(stats), nparts, static_cast<float2*>(rowstats), rows);
  return cudaGetLastError();
}

cudaError_t launch_row_dot(const void* dO, const void* O, float* D, int64_t b, int64_t s, int64_t h, int heads,
                           cudaStream_t stream, int num_sms) {
  (void)num_sms;
  const int64_t n = b * s;  // token rows, one warp each
  if (n <= 0) return cudaSuccess;
  if ((h / heads) % 8 != 0) return cudaErrorInvalidValue;
  row_dot_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), D, b, s, h, heads);
  return cudaGetLastError();
}


}  // namespace tpmlp
