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

// Where a LayerNorm writes its output row: in place of the input row, or, for the sequence-parallel
// block, at the row's token-order position (the all-gather g fused into the LayerNorm's store).
struct LnOutRows {
  int64_t b, s, sl;  // sl = 0: the input row's own position
  __device__ __forceinline__ int64_t operator()(int64_t R) const {
    return sl ? shard_row_to_token(R, b, s, sl) : R;
  }
};

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
                                                               T* __restrict__ y, int64_t rows, int h,
                                                               LnOutRows out_rows) {
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
    T* yr = y + out_rows(r) * h;
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
                                                                T* __restrict__ y, int64_t rows, int64_t h,
                                                                LnOutRows out_rows) {
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
    T* yr = y + out_rows(r) * h;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x)
      yr[c] = static_cast<T>(fmaf((static_cast<float>(xr[c]) - mean) * rstd, gamma[c], beta[c]));
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
// rare cases redo the vector in full. Each thread stores its vector's 8 mask bits as one byte
// of the mask words. kLow3 = seed & 7.
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
      // The vector's 8 mask bits are byte k0 / 8 of the little-endian mask words (bit k of word
      // k / 32): one byte store per thread, the warp's 32 bytes contiguous.
      if (mask_bits != nullptr && v < nvec)
        reinterpret_cast<uint8_t*>(mask_bits)[(flat_row + static_cast<uint64_t>(v) * 8) >> 3] = static_cast<uint8_t>(bits);
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
                            float eps, T* __restrict__ y, int64_t rows, int h, unsigned int* status,
                            LnOutRows out_rows) {
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
    T* yr = y + out_rows(R) * h;
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
        for (uint32_t e = 0; e < 8; e += 2) {  // pairs: g * scale on the f32x2 path
          const uint32_t c0 = hs.high(e), c1 = hs.high(e + 1);
          redo |= (c0 == hs.thi) | (c1 == hs.thi);
          const float2 f = f2_split(f2_mul(f2_make(gf[e], gf[e + 1]), f2_make(scale, scale)));
          o[e] = c0 < hs.thi ? 0.f : f.x;
          o[e + 1] = c1 < hs.thi ? 0.f : f.y;
        }
        Vec8<T> ov;
        ov.from_float(o);
        ov.store(dst + v * 8);
      }
      if (redo) dropout_vector_full<T>(src + v * 8, nullptr, dst + v * 8, base, threshold, scale);
    }
  }
}

// 8 elements of T as four fp32 pairs, and back.
__device__ __forceinline__ void to_f2(const uint4& u, F2 (&o)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = f2_make(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
__device__ __forceinline__ void to_f2(const float4 (&u)[2], F2 (&o)[4]) {
  o[0] = f2_make(u[0].x, u[0].y);
  o[1] = f2_make(u[0].z, u[0].w);
  o[2] = f2_make(u[1].x, u[1].y);
  o[3] = f2_make(u[1].z, u[1].w);
}
__device__ __forceinline__ void from_f2(const F2 (&o)[4], uint4& u) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = f2_split(o[i]);
    w[i] = pack_bf16x2(p.x, p.y);
  }
  u = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void from_f2(const F2 (&o)[4], float4 (&u)[2]) {
  const float2 a = f2_split(o[0]), b = f2_split(o[1]), c = f2_split(o[2]), d = f2_split(o[3]);
  u[0] = make_float4(a.x, a.y, b.x, b.y);
  u[1] = make_float4(c.x, c.y, d.x, d.y);
}

// One vector of 8 elements as it sits in registers: a uint4 of bf16 pairs, or two float4.
template <typename T>
struct Raw8 {
  uint4 u;
  __device__ __forceinline__ void load(const T* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void store(T* p) const { *reinterpret_cast<uint4*>(p) = u; }
  __device__ __forceinline__ void unpack(F2 (&o)[4]) const { to_f2(u, o); }
  __device__ __forceinline__ void pack(const F2 (&o)[4]) { from_f2(o, u); }
};
template <>
struct Raw8<float> {
  float4 u[2];
  __device__ __forceinline__ void load(const float* p) {
    u[0] = reinterpret_cast<const float4*>(p)[0];
    u[1] = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void store(float* p) const {
    reinterpret_cast<float4*>(p)[0] = u[0];
    reinterpret_cast<float4*>(p)[1] = u[1];
  }
  __device__ __forceinline__ void unpack(F2 (&o)[4]) const { to_f2(u, o); }
  __device__ __forceinline__ void pack(const F2 (&o)[4]) { from_f2(o, u); }
};

// The same dropout backward with the forward's mask bits read back instead of recomputed (bit i
// of word w set iff element 32 w + i of the token-order tensor was dropped; rows of h % 32 == 0
// columns start on a word): a gather with a bit test, one thread per vector of 8 elements.
template <typename T>
__global__ void __launch_bounds__(128) dropout_grad_gather_mask_kernel(const T* __restrict__ dout,
                                                                       T* __restrict__ dtok,
                                                                       const uint32_t* __restrict__ mask_bits,
                                                                       float scale, int64_t rows, int64_t b,
                                                                       int64_t s, int64_t sl, int h) {
  const int nvec = h >> 3;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* src = dout + token_to_shard_row(r, b, s, sl) * h;
    T* dst = dtok + r * h;
    const uint32_t* mrow = mask_bits + ((static_cast<uint64_t>(r) * static_cast<uint64_t>(h)) >> 5);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      Vec8<T> gv;
      gv.load(src + v * 8);
      const uint32_t bits = __ldg(mrow + (v >> 2)) >> ((v & 3) * 8);
      float gf[8], o[8];
      gv.to_float(gf);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (bits >> e) & 1u ? 0.f : gf[e] * scale;
      Vec8<T> ov;
      ov.from_float(o);
      ov.store(dst + v * 8);
    }
  }
}

// LayerNorm backward (or RMSNorm's, kRms) with an optional residual gradient dres (kRes), for
// rows of up to 8192 columns ("Megatron 训练" notes, section "LayerNorm"; the SP backward chain
// of the "Efficient Large-Scale ... Megatron-LM" notes, section 3.5.1):
//   LN : dx = dres + rstd * (g - mean(g) - x_hat * mean(g * x_hat)),   x_hat = (x - mu) * rstd
//   RMS: dx = dres + rstd * (g - x_hat * mean(g * x_hat)),              x_hat = x * rstd
// with g = dy * gamma; dgamma = sum over rows of dy * x_hat, dbeta = sum over rows of dy.
// Rows stream through a shared-memory ring of bulk copies (CTA c takes rows c + i * gridDim.x).
// R rows are processed per step: each of the NT threads owns CH vectors of 8 columns, reads
// its columns of the R rows out of the ring into registers, adds its share of the row sums
// (sum d, d^2, g, g*d with d = x - x_0 for LayerNorm; d^2 and g*d for RMSNorm), and the warps'
// sums meet in shared memory behind one barrier per step; the ring stages are then refilled at
// once, since the data is in registers. Every warp adds the per-warp sums in the same order
// (deterministic), the row's coefficients follow, and the second pass writes dx and adds dgamma,
// dbeta into registers, which go to partials[blockIdx][2][h] at the end for a fixed-order sum
// (sum_partials_kernel, launched as this grid's programmatic dependent).
// The elementwise arithmetic runs on fp32 pairs (f32x2). Every wait is bounded; on a timeout the
// CTA stops after the step's barrier, thread 0 waits (bounded) for its copies and the CTA returns.
template <typename T, int NT, int CH, int R, bool kRms, bool kRes, int MINB = 0>
__global__ void __launch_bounds__(NT, MINB)
    norm_backward_kernel(const T* __restrict__ x, const T* __restrict__ dy, const T* __restrict__ dres,
                         const float* __restrict__ gamma, float eps, T* __restrict__ dx,
                         float* __restrict__ partials, int64_t rows, int h, int stages, unsigned int* status) {
  constexpr int NW = NT / 32;
  constexpr int NTEN = kRes ? 3 : 2;  // tensors staged per row: x, dy (, dres)
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float4 red[2][R][NW];
  __shared__ int s_abort;
  const uint32_t row_bytes = static_cast<uint32_t>(h) * sizeof(T);
  const uint32_t stage_bytes = NTEN * row_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(stages) * stage_bytes);
  const int64_t nloc = rows_for_cta(rows);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  auto issue = [&](int64_t i) {
    const int64_t row = blockIdx.x + i * gridDim.x;
    const int st = static_cast<int>(i % stages);
    uint8_t* dst = smem + static_cast<size_t>(st) * stage_bytes;
    mbar_arrive_expect_tx(&full[st], stage_bytes);
    bulk_load(dst, x + row * h, row_bytes, &full[st]);
    bulk_load(dst + row_bytes, dy + row * h, row_bytes, &full[st]);
    if constexpr (kRes) bulk_load(dst + 2 * row_bytes, dres + row * h, row_bytes, &full[st]);
  };
  int64_t issued = nloc < stages ? nloc : stages;  // meaningful in thread 0 only
  if (tid == 0)
    for (int64_t i = 0; i < issued; ++i) issue(i);

  F2 gam[CH][4], accg[CH][4], accb[kRms ? 1 : CH][4];
  const F2 zero = f2_make(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int col = (tid + c * NT) * 8;
    float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
    if (col < h) {
      g0 = *reinterpret_cast<const float4*>(gamma + col);
      g1 = *reinterpret_cast<const float4*>(gamma + col + 4);
    }
    gam[c][0] = f2_make(g0.x, g0.y);
    gam[c][1] = f2_make(g0.z, g0.w);
    gam[c][2] = f2_make(g1.x, g1.y);
    gam[c][3] = f2_make(g1.z, g1.w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      accg[c][e] = zero;
      if constexpr (!kRms) accb[c][e] = zero;
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);

  int64_t i0 = 0;
  for (; i0 < nloc; i0 += R) {
    const int par = static_cast<int>((i0 / R) & 1);
    Raw8<T> xv[R][CH], dv[R][CH], rv[kRes ? R : 1][CH];
    float shift[R];
    float4 part[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      part[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      shift[j] = 0.f;
      const int64_t i = i0 + j;
      if (i >= nloc) continue;  // the same for every thread of the CTA
      const int st = static_cast<int>(i % stages);
      if (!mbar_wait(&full[st], static_cast<uint32_t>((i / stages) & 1), status, 23)) s_abort = 1;
      const T* xs = reinterpret_cast<const T*>(smem + static_cast<size_t>(st) * stage_bytes);
      const T* ds = reinterpret_cast<const T*>(smem + static_cast<size_t>(st) * stage_bytes + row_bytes);
      if constexpr (!kRms) shift[j] = static_cast<float>(xs[0]);
      const F2 sh = f2_make(shift[j], shift[j]);
      F2 s_d = zero, s_dd = zero, s_g = zero, s_gd = zero;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int col = (tid + c * NT) * 8;
        if (col < h) {
          xv[j][c].load(xs + col);
          dv[j][c].load(ds + col);
          if constexpr (kRes) {
            const T* rs = reinterpret_cast<const T*>(smem + static_cast<size_t>(st) * stage_bytes + 2 * row_bytes);
            rv[j][c].load(rs + col);
          }
          F2 xf[4], df[4];
          xv[j][c].unpack(xf);
          dv[j][c].unpack(df);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const F2 d = kRms ? xf[e] : f2_sub(xf[e], sh);
            const F2 g = f2_mul(df[e], gam[c][e]);
            if constexpr (!kRms) {
              s_d = f2_add(s_d, d);
              s_g = f2_add(s_g, g);
            }
            s_dd = f2_fma(d, d, s_dd);
            s_gd = f2_fma(g, d, s_gd);
          }
        }
      }
      const float2 a = f2_split(s_d), b = f2_split(s_dd), c2 = f2_split(s_g), d2 = f2_split(s_gd);
      part[j] = make_float4(a.x + a.y, b.x + b.y, c2.x + c2.y, d2.x + d2.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if constexpr (!kRms) {
          part[j].x += __shfl_xor_sync(0xffffffffu, part[j].x, o);
          part[j].z += __shfl_xor_sync(0xffffffffu, part[j].z, o);
        }
        part[j].y += __shfl_xor_sync(0xffffffffu, part[j].y, o);
        part[j].w += __shfl_xor_sync(0xffffffffu, part[j].w, o);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < R; ++j) red[par][j][w] = part[j];
    }
    __syncthreads();  // every thread has its rows' data in registers and the warps' sums are out
    if (s_abort) break;
    if (tid == 0) {
      for (int64_t i = i0; i < i0 + R && i < nloc; ++i)
        if (i + stages < nloc) {
          issue(i + stages);
          issued = i + stages + 1;
        }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int64_t i = i0 + j;
      if (i >= nloc) continue;
      // Every warp adds the NW per-warp sums in the same order: lanes k < NW hold sum k, a
      // butterfly over log2(NW) lanes adds them, lane 0's total is broadcast.
      float4 v = lane < NW ? red[par][j][lane] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int o = 1; o < NW; o <<= 1) {
        if constexpr (!kRms) {
          v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
          v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
        }
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
      }
      float sd = 0.f, sg = 0.f;
      if constexpr (!kRms) {
        sd = __shfl_sync(0xffffffffu, v.x, 0);
        sg = __shfl_sync(0xffffffffu, v.z, 0);
      }
      const float sdd = __shfl_sync(0xffffffffu, v.y, 0);
      const float sgd = __shfl_sync(0xffffffffu, v.w, 0);
      const float md = sd * inv_h;                                          // mean(x) - x_0 (0 for RMS)
      const float rstd = rsqrtf((kRms ? sdd * inv_h : fmaxf(sdd * inv_h - md * md, 0.f)) + eps);
      const float mean_g = sg * inv_h;                                      // 0 for RMS
      const float mean_gxh = rstd * (sgd * inv_h - md * mean_g);            // mean(g * x_hat)
      const float nmu_r = -(shift[j] + md) * rstd;                          // x_hat = x * rstd + nmu_r
      const float k1 = -rstd * mean_gxh * rstd;                             // dx = rstd*g + k1*x + k0 (+ dres)
      const float k0 = -rstd * mean_g + (-rstd * mean_gxh) * nmu_r;
      const F2 r2 = f2_make(rstd, rstd), nm2 = f2_make(nmu_r, nmu_r), k1_2 = f2_make(k1, k1),
               k0_2 = f2_make(k0, k0);
      T* outr = dx + (blockIdx.x + i * gridDim.x) * h;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int col = (tid + c * NT) * 8;
        if (col < h) {
          F2 xf[4], df[4], o[4];
          xv[j][c].unpack(xf);
          dv[j][c].unpack(df);
          F2 rf[4];
          if constexpr (kRes) rv[j][c].unpack(rf);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const F2 xh = f2_fma(xf[e], r2, nm2);
            accg[c][e] = f2_fma(df[e], xh, accg[c][e]);
            if constexpr (!kRms) accb[c][e] = f2_add(accb[c][e], df[e]);
            F2 t = f2_fma(k1_2, xf[e], k0_2);
            if constexpr (kRes) t = f2_add(t, rf[e]);
            o[e] = f2_fma(r2, f2_mul(df[e], gam[c][e]), t);
          }
          Raw8<T> ov;
          ov.pack(o);
          ov.store(outr + col);
        }
      }
    }
  }
  // Lets the dependent partial-sum grid be scheduled; it still waits for this grid to complete.
  asm volatile("griddepcontrol.launch_dependents;");
  if (s_abort && tid == 0) {
    // Copies that may still be in flight: the rows of the step that gave up and every row
    // issued after them (each is the next phase of its own stage).
    for (int64_t k = i0; k < issued; ++k) mbar_wait(&full[k % stages], (k / stages) & 1, status, 21);
  }
  float* pg = partials + static_cast<int64_t>(blockIdx.x) * 2 * h;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int col = (tid + c * NT) * 8;
    if (col < h) {
      float2 gq[4], bq[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gq[e] = f2_split(accg[c][e]);
        bq[e] = kRms ? make_float2(0.f, 0.f) : f2_split(accb[kRms ? 0 : c][e]);
      }
      reinterpret_cast<float4*>(pg + col)[0] = make_float4(gq[0].x, gq[0].y, gq[1].x, gq[1].y);
      reinterpret_cast<float4*>(pg + col)[1] = make_float4(gq[2].x, gq[2].y, gq[3].x, gq[3].y);
      reinterpret_cast<float4*>(pg + h + col)[0] = make_float4(bq[0].x, bq[0].y, bq[1].x, bq[1].y);
      reinterpret_cast<float4*>(pg + h + col)[1] = make_float4(bq[2].x, bq[2].y, bq[3].x, bq[3].y);
    }
  }

}

// dgamma[c] = sum over CTAs k of partials[k][0][c], dbeta[c] likewise from partials[k][1][c]. A
// CTA of 1024 threads takes kSumPartialsCols = 32 columns: thread (g, q) adds the float4 of columns
// 4q..4q+3 over partials g, g + 128, g + 256, ... (a few loads each, all in flight); the 128 group
// sums are then added by a fixed pairwise tree, so the result does not depend on scheduling. With
// dbeta null only the dgamma half is read. Narrow column slices give enough CTAs to cover the SMs
// (128 for h = 4096), since the work is latency-bound. Launched as a programmatic dependent of the
// norm backward kernel, it waits (griddepcontrol.wait) for that grid's completion and memory.
constexpr int kSumPartialsThreads = 1024;
constexpr int kSumPartialsCols = 32;
__global__ void __launch_bounds__(kSumPartialsThreads)
    sum_partials_kernel(const float* __restrict__ partials, int nparts, int h, float* __restrict__ dgamma,
                        float* __restrict__ dbeta) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kQuads = kSumPartialsCols / 4;                  // 8
  constexpr int kGroups = kSumPartialsThreads / kQuads;         // 128
  __shared__ float4 grp[kGroups][kQuads];
  const int q = threadIdx.x % kQuads, g = threadIdx.x / kQuads;
  const int ncols = dbeta ? 2 * h : h;
  const int c = blockIdx.x * kSumPartialsCols + q * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < ncols) {
    const float* p = partials + c;
#pragma unroll 8
    for (int k = g; k < nparts; k += kGroups) {
      const float4 v = *reinterpret_cast<const float4*>(p + static_cast<int64_t>(k) * 2 * h);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
  }
  grp[g][q] = acc;
#pragma unroll
  for (int half = kGroups / 2; half > 0; half >>= 1) {
    __syncthreads();
    if (g < half) {
      const float4 o = grp[g + half][q];
      acc.x += o.x;
      acc.y += o.y;
      acc.z += o.z;
      acc.w += o.w;
      grp[g][q] = acc;
    }
  }
  if (g == 0 && c < ncols) {
    if (c < h) *reinterpret_cast<float4*>(dgamma + c) = acc;
    else *reinterpret_cast<float4*>(dbeta + (c - h)) = acc;
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
// and L = sum_j l_j * 2^(m_j - M), stored as (M + log2 L, 1/L). A warp takes 32 rows: chunks of
// 16 partials (128 bytes of each row) are read line-wide (4 rows x 128 bytes per instruction)
// into the warp's shared-memory block (16-byte segments XOR-swizzled by row), each lane then
// takes its own row out of it and folds the chunk into a running (M, L) in index order.
__global__ void __launch_bounds__(256) softmax_combine_kernel(const float2* __restrict__ stats, int nparts,
                                                              float2* __restrict__ rowstats, int64_t rows) {
  __shared__ __align__(16) uint8_t sbuf[8][32 * 128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = (static_cast<int64_t>(blockIdx.x) * 8 + warp) * 32;
  if (r0 >= rows) return;  // uniform across the warp
  uint8_t* buf = sbuf[warp];
  const uint8_t* base = reinterpret_cast<const uint8_t*>(stats);
  const int64_t row_bytes = static_cast<int64_t>(nparts) * 8;
  float M = -INFINITY, L = 0.f;
  for (int c = 0; c * 16 < nparts; ++c) {
    const int segs = min(8, (nparts - c * 16) / 2);  // 16-byte segments of this chunk in a row
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3), j = lane & 7;
      float4 v = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      if (r0 + rr < rows && j < segs)
        v = *reinterpret_cast<const float4*>(base + (r0 + rr) * row_bytes + c * 128 + j * 16);
      *reinterpret_cast<float4*>(buf + rr * 128 + ((j ^ (rr & 7)) << 4)) = v;
    }
    __syncwarp();
    float4 mine[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) mine[j] = *reinterpret_cast<const float4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4));
    __syncwarp();
    float mc = M;
#pragma unroll
    for (int j = 0; j < 8; ++j) mc = fmaxf(mc, fmaxf(mine[j].x, mine[j].z));
    float lc = L > 0.f ? L * ex2_approx(M - mc) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      lc += mine[j].y > 0.f ? mine[j].y * ex2_approx(mine[j].x - mc) : 0.f;
      lc += mine[j].w > 0.f ? mine[j].w * ex2_approx(mine[j].z - mc) : 0.f;
    }
    M = mc;
    L = lc;
  }
  // the softmax pass needs only M + log2(L): P = 2^(y - M) / L = 2^(y - (M + log2 L))
  if (r0 + lane < rows) rowstats[r0 + lane] = make_float2(M + log2f(L), 1.0f / L);
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

// The same row dot products for dh / 8 dividing 32, heads <= kRowDotMaxHeads and s % 8 == 0: a
// CTA takes 8 consecutive tokens of one sequence (a warp each). A warp issues the loads of eight
// head groups before it reduces any (the groups' loads in flight together instead of one group's
// at a time), and the CTA's results go through shared memory so that each head's 8 values are
// stored as one 32-byte segment instead of 8 scattered words.
constexpr int kRowDotMaxHeads = 128;
__global__ void __launch_bounds__(256) row_dot_staged_kernel(const __nv_bfloat16* __restrict__ dO,
                                                             const __nv_bfloat16* __restrict__ O,
                                                             float* __restrict__ D, int64_t s, int64_t h,
                                                             int heads) {
  __shared__ float sd[8][kRowDotMaxHeads];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok0 = static_cast<int64_t>(blockIdx.x) * 8;
  const int64_t tok = tok0 + w;
  const int64_t dh = h / heads;
  const int vh = static_cast<int>(dh / 8);
  const int hpw = 32 / vh, seg = lane / vh, v = lane % vh;
  const __nv_bfloat16* a = dO + tok * h;
  const __nv_bfloat16* c = O + tok * h;
  constexpr int kGroups = 8;
  for (int j0 = 0; j0 < heads; j0 += kGroups * hpw) {
    uint4 va[kGroups], vc[kGroups];
#pragma unroll
    for (int u = 0; u < kGroups; ++u) {
      const int j = j0 + u * hpw + seg;
      if (j < heads) {
        va[u] = *reinterpret_cast<const uint4*>(a + j * dh + v * 8);
        vc[u] = *reinterpret_cast<const uint4*>(c + j * dh + v * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroups; ++u) {
      const int j = j0 + u * hpw + seg;
      float acc = 0.f;
      if (j < heads) {
        const uint32_t wa[4] = {va[u].x, va[u].y, va[u].z, va[u].w};
        const uint32_t wc[4] = {vc[u].x, vc[u].y, vc[u].z, vc[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 fa = unpack_bf16x2(wa[k]), fc = unpack_bf16x2(wc[k]);
          acc = fmaf(fa.x, fc.x, acc);
          acc = fmaf(fa.y, fc.y, acc);
        }
      }
      for (int o = vh / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (v == 0 && j < heads) sd[w][j] = acc;
    }
  }
  __syncthreads();
  const int64_t bi = tok0 / s, si0 = tok0 - bi * s;
  for (int idx = threadIdx.x; idx < 8 * heads; idx += blockDim.x) {
    const int j = idx >> 3, t = idx & 7;
    D[(bi * heads + j) * s + si0 + t] = sd[t][j];
  }
}

int rows_grid(int64_t rows, int num_sms, int per_sm) {
  const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
  return static_cast<int>(rows < cap ? (rows > 0 ? rows : 1) : cap);
}

}  // namespace

cudaError_t launch_layernorm(const void* x, const float* gamma, const float* beta, float eps, void* y, int64_t rows,
                             int64_t h, bool bf16, cudaStream_t stream, int num_sms, unsigned int* status, bool rms,
                             const int64_t* gather_bst) {
  if (rows <= 0) return cudaSuccess;
  LnOutRows out_rows{0, 0, 0};
  if (gather_bst) out_rows = LnOutRows{gather_bst[0], gather_bst[1], gather_bst[1] / gather_bst[2]};
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
                                                   static_cast<TYPE*>(y), rows, (int)h, status, out_rows);      \
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
      if (ch <= 1) layernorm_kernel<__nv_bfloat16, 1><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
      else if (ch <= 2) layernorm_kernel<__nv_bfloat16, 2><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
      else if (ch <= 4) layernorm_kernel<__nv_bfloat16, 4><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
      else layernorm_kernel<__nv_bfloat16, 8><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
    } else {
      auto xp = static_cast<const float*>(x);
      auto yp = static_cast<float*>(y);
      if (ch <= 1) layernorm_kernel<float, 1><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
      else if (ch <= 2) layernorm_kernel<float, 2><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
      else if (ch <= 4) layernorm_kernel<float, 4><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
      else layernorm_kernel<float, 8><<<grid, kLnThreads, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h, out_rows);
    }
  } else {
    const int grid = rows_grid(rows, num_sms, 8);
    if (bf16)
      layernorm_generic_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), gamma, beta, eps, static_cast<__nv_bfloat16*>(y), rows, h, out_rows);
    else
      layernorm_generic_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), gamma, beta, eps,
                                                                 static_cast<float*>(y), rows, h, out_rows);
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

cudaError_t launch_dropout_grad_gather(const void* dout_shards, void* dtok, const uint32_t* mask_bits,
                                       uint64_t threshold, float scale, uint64_t seed, int64_t b, int64_t s,
                                       int64_t h, int t, bool bf16, cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0 || (mask_bits && h % 32 != 0)) return cudaErrorInvalidValue;
  const int grid = rows_grid(rows, num_sms, 64);  // one row per CTA up to 64 CTAs per SM
  if (mask_bits) {
    if (bf16)
      dropout_grad_gather_mask_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(dout_shards), static_cast<__nv_bfloat16*>(dtok), mask_bits, scale, rows,
          b, s, s / t, static_cast<int>(h));
    else
      dropout_grad_gather_mask_kernel<float><<<grid, 128, 0, stream>>>(static_cast<const float*>(dout_shards),
                                                                       static_cast<float*>(dtok), mask_bits, scale,
                                                                       rows, b, s, s / t, static_cast<int>(h));
    return cudaGetLastError();
  }
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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared memory a norm_backward_kernel CTA may fill with ring stages.
constexpr size_t kNormBwdSmemBudget = 200 * 1024;

// One launch of norm_backward_kernel with `stages` ring stages; the grid is one resident wave (as
// many CTAs as fit on the SMs at once), at most kLnBwdMaxCtas (the partials' capacity). Then the
// partial sums, as a programmatic dependent launch: its CTAs may be scheduled while the norm
// kernel's last CTAs finish, and wait in griddepcontrol.wait for that grid to complete.
template <typename T, int NT, int CH, int R, bool kRms, bool kRes, int MINB = 0>
cudaError_t launch_norm_bwd(const void* x, const void* dy, const void* dres, const float* gamma, float eps, void* dx,
                            float* partials, float* dgamma, float* dbeta, int64_t rows, int h, int stages,
                            int num_sms, cudaStream_t stream, unsigned int* status) {
  auto k = norm_backward_kernel<T, NT, CH, R, kRms, kRes, MINB>;
  const size_t stage_bytes = (kRes ? 3 : 2) * static_cast<size_t>(h) * sizeof(T);
  const size_t smem = staged_smem(stage_bytes, stages);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, NT, smem) != cudaSuccess || per_sm < 1) per_sm = 1;
  int grid = rows_grid(rows, num_sms, per_sm);
  grid = grid < kLnBwdMaxCtas ? grid : kLnBwdMaxCtas;
  k<<<grid, NT, smem, stream>>>(static_cast<const T*>(x), static_cast<const T*>(dy), static_cast<const T*>(dres),
                                gamma, eps, static_cast<T*>(dx), partials, rows, h, stages, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int ncols = dbeta ? 2 * h : h;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((ncols + kSumPartialsCols - 1) / kSumPartialsCols), 1, 1);
  cfg.blockDim = dim3(kSumPartialsThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sum_partials_kernel, static_cast<const float*>(partials), grid, h, dgamma, dbeta);
}

// Threads per CTA and vectors per thread by width: at most 16 columns per thread, at least 128
// threads; one row per step; three ring stages per CTA (or fewer for wide fp32 rows), so that
// two or three CTAs share an SM.
template <typename T, bool kRms, bool kRes>
cudaError_t launch_norm_bwd_for_width(const void* x, const void* dy, const void* dres, const float* gamma, float eps,
                                      void* dx, float* partials, float* dgamma, float* dbeta, int64_t rows, int h,
                                      int num_sms, cudaStream_t stream, unsigned int* status) {
  const size_t stage_bytes = (kRes ? 3 : 2) * static_cast<size_t>(h) * sizeof(T);
  int stages = static_cast<int>(kNormBwdSmemBudget / (stage_bytes + sizeof(uint64_t)));
  stages = stages > 3 ? 3 : stages;  // >= 2: a stage holds at most 3 x 8192 x 4 bytes = 96 KiB
  if (h <= 1024)
    return launch_norm_bwd<T, 128, 1, 1, kRms, kRes>(x, dy, dres, gamma, eps, dx, partials, dgamma, dbeta, rows, h,
                                                     stages, num_sms, stream, status);
  if (h <= 2048)
    return launch_norm_bwd<T, 128, 2, 1, kRms, kRes>(x, dy, dres, gamma, eps, dx, partials, dgamma, dbeta, rows, h,
                                                     stages, num_sms, stream, status);
  if (h <= 4096)
    return launch_norm_bwd<T, 256, 2, 1, kRms, kRes>(x, dy, dres, gamma, eps, dx, partials, dgamma, dbeta, rows, h,
                                                     stages, num_sms, stream, status);
  return launch_norm_bwd<T, 512, 2, 1, kRms, kRes>(x, dy, dres, gamma, eps, dx, partials, dgamma, dbeta, rows, h,
                                                   stages, num_sms, stream, status);
}

cudaError_t launch_layernorm_backward(const void* x, const void* dxn, const void* dout, const float* gamma, float eps,
                                      void* dx, float* partials, float* dgamma, float* dbeta, int64_t rows, int64_t h,
                                      bool bf16, cudaStream_t stream, int num_sms, bool rms, unsigned int* status) {
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0 || h > kNormBwdMaxH || !aligned16(x) || !aligned16(dxn) || !aligned16(dx) ||
      (dout && !aligned16(dout)) || (rms && dout) || (!rms && !dbeta) || !aligned16(dgamma) ||
      (dbeta && !aligned16(dbeta)))
    return cudaErrorInvalidValue;
  const int hi = static_cast<int>(h);
  if (bf16) {
    using T = __nv_bfloat16;
    if (rms) return launch_norm_bwd_for_width<T, true, false>(x, dxn, nullptr, gamma, eps, dx, partials, dgamma,
                                                              nullptr, rows, hi, num_sms, stream, status);
    if (dout) return launch_norm_bwd_for_width<T, false, true>(x, dxn, dout, gamma, eps, dx, partials, dgamma, dbeta,
                                                               rows, hi, num_sms, stream, status);
    return launch_norm_bwd_for_width<T, false, false>(x, dxn, nullptr, gamma, eps, dx, partials, dgamma, dbeta, rows,
                                                      hi, num_sms, stream, status);
  }
  using T = float;
  if (rms) return launch_norm_bwd_for_width<T, true, false>(x, dxn, nullptr, gamma, eps, dx, partials, dgamma, nullptr,
                                                            rows, hi, num_sms, stream, status);
  if (dout) return launch_norm_bwd_for_width<T, false, true>(x, dxn, dout, gamma, eps, dx, partials, dgamma, dbeta,
                                                             rows, hi, num_sms, stream, status);
  return launch_norm_bwd_for_width<T, false, false>(x, dxn, nullptr, gamma, eps, dx, partials, dgamma, dbeta, rows, hi,
                                                    num_sms, stream, status);
}

cudaError_t launch_softmax_combine(const void* stats, int nparts, void* rowstats, int64_t rows, cudaStream_t stream,
                                   int num_sms) {
  (void)num_sms;
  if (rows <= 0) return cudaSuccess;
  if (nparts > 64 || nparts % 2 != 0) return cudaErrorInvalidValue;  // s <= 8192: at most 2 * 32 parts
  softmax_combine_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, stream>>>(  // 8 warps x 32 rows
      static_cast<const float2*>(stats), nparts, static_cast<float2*>(rowstats), rows);
  return cudaGetLastError();
}

cudaError_t launch_row_dot(const void* dO, const void* O, float* D, int64_t b, int64_t s, int64_t h, int heads,
                           cudaStream_t stream, int num_sms) {
  (void)num_sms;
  const int64_t n = b * s;  // token rows, one warp each
  if (n <= 0) return cudaSuccess;
  if ((h / heads) % 8 != 0) return cudaErrorInvalidValue;
  const int64_t vh = h / heads / 8;
  if (vh <= 32 && 32 % vh == 0 && heads <= kRowDotMaxHeads && s % 8 == 0) {
    row_dot_staged_kernel<<<static_cast<unsigned>(n / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), D, s, h, heads);
    return cudaGetLastError();
  }
  row_dot_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(O), D, b, s, h, heads);
  return cudaGetLastError();
}


}  // namespace tpmlp
