// Merge of split-KV partial outputs by their log-sum-exp (MLA DCP decode study
// notes, section 1.1: partials merged by LSE equal one softmax over the whole
// sequence).
//
// Many rows: a group of LPR lanes owns one (token, head) row; every lane moves
// 16-byte vectors, so a row of D bf16 values is read with D*2/16 lanes in one
// coalesced sweep per partition, two partitions' loads in flight at once.  Few
// rows: one warp per row with all partitions in flight (below).  Partitions
// whose LSE is -inf are skipped before their output is touched, so their
// (unwritten) rows are never read.
#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr int kThreads = 256;
// Partitions whose loads are issued together.  Two keep DRAM busy; eight
// concurrent streams, 2^k bytes apart, measured 40% slower than two.
constexpr int kBatch = 2;

template <typename T, int D>
struct CombineShape {
  static constexpr int kVecElems = 16 / sizeof(T);            // elements per 16-byte vector
  static constexpr int kVecs = D / kVecElems;                  // vectors per row
  static constexpr int kLpr = kVecs < 32 ? kVecs : 32;         // lanes per row
  static constexpr int kVpl = kVecs / kLpr;                    // vectors per lane
  static constexpr int kRowsPerWarp = 32 / kLpr;
};

template <typename T>
__device__ inline void accum(float *acc, const uint4 &v, float w) {
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
    }
  } else {
    const float *f = reinterpret_cast<const float *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf(w, f[i], acc[i]);
  }
}

template <typename T>
__device__ inline uint4 pack(const float *x) {
  uint4 r;
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
  } else {
    float *f = reinterpret_cast<float *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = x[i];
  }
  return r;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
lse_combine_kernel(const T *__restrict__ po, const float *__restrict__ pl, int32_t num_splits,
                   int64_t rows, T *__restrict__ out, float *__restrict__ out_lse) {
  using Sh = CombineShape<T, D>;
  constexpr int E = Sh::kVecElems;
  pdl_wait();                                                // the partials' producer is done
  const int lane = threadIdx.x & 31;
  const int sub = lane / Sh::kLpr;              // row within the warp
  const int gl = lane % Sh::kLpr;               // lane within the row group
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t row = warp * Sh::kRowsPerWarp + sub;
  const bool live = row < rows;

  // 1) L = max_p lse_p over the group's lanes
  float L = -INFINITY;
  if (live)
    for (int p = gl; p < num_splits; p += Sh::kLpr) L = fmaxf(L, __ldg(pl + (int64_t)p * rows + row));
#pragma unroll
  for (int o = Sh::kLpr / 2; o > 0; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));  // stays inside the group

  float acc[Sh::kVpl * E];
#pragma unroll
  for (int i = 0; i < Sh::kVpl * E; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (live && L != -INFINITY) {
    // partitions in batches of kBatch: every load of a batch is in flight
    // before the first multiply-add
    for (int p0 = 0; p0 < num_splits; p0 += kBatch) {
      float w[kBatch];
      uint4 v[kBatch][Sh::kVpl];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int p = p0 + i;
        const float lp = p < num_splits ? __ldg(pl + (int64_t)p * rows + row) : -INFINITY;
        w[i] = lp == -INFINITY ? 0.f : __expf(lp - L);      // lp <= L: an argument in (-inf, 0]
        const uint4 *src = reinterpret_cast<const uint4 *>(po + ((int64_t)p * rows + row) * D);
#pragma unroll
        for (int j = 0; j < Sh::kVpl; ++j)
          v[i][j] = w[i] > 0.f ? __ldg(src + gl + j * Sh::kLpr) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        wsum += w[i];
#pragma unroll
        for (int j = 0; j < Sh::kVpl; ++j) accum<T>(acc + j * E, v[i][j], w[i]);
      }
    }
  }
  if (!live) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int i = 0; i < Sh::kVpl * E; ++i) acc[i] *= inv;
  uint4 *dst = reinterpret_cast<uint4 *>(out + row * D);
#pragma unroll
  for (int v = 0; v < Sh::kVpl; ++v) dst[gl + v * Sh::kLpr] = pack<T>(acc + v * E);
  if (out_lse != nullptr && gl == 0) out_lse[row] = (wsum > 0.f) ? L + logf(wsum) : -INFINITY;
}

// Few rows (a decode step: tokens x heads in the thousands) leave too little
// work in flight for the kernel above, whose partitions follow one another.
// Here one warp owns a row: the lanes read the partitions' LSEs for the
// maximum, then split into kGroups groups that each take every kGroups-th
// partition, a batch of partitions' vectors in flight before the first
// multiply-add; the groups' sums meet through shuffles.
template <typename T, int D>
struct RowWarpShape {
  static constexpr int kVecElems = 16 / sizeof(T);
  static constexpr int kVecs = D / kVecElems;                 // 16-byte vectors per row
  static constexpr int kLanes = kVecs < 32 ? kVecs : 32;      // lanes per partition group
  static constexpr int kGroups = 32 / kLanes;
  static constexpr int kVpl = kVecs / kLanes;                 // vectors per lane and partition
  // partitions per lane per batch: up to 32 partitions per batch, at most 8
  // vectors per lane in flight (more measured slower at the decode size)
  static constexpr int kInFlight = 32 / kGroups < 8 / kVpl ? 32 / kGroups : 8 / kVpl;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
lse_combine_rowwarp_kernel(const T *__restrict__ po, const float *__restrict__ pl, int32_t num_splits,
                           int64_t rows, T *__restrict__ out, float *__restrict__ out_lse) {
  using Sh = RowWarpShape<T, D>;
  constexpr int E = Sh::kVecElems;
  pdl_wait();                                                // the partials' producer is done
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  if (row >= rows) return;                                   // warp-uniform
  const int g = lane / Sh::kLanes, gl = lane % Sh::kLanes;
  float L = -INFINITY;
  for (int p = lane; p < num_splits; p += 32) L = fmaxf(L, __ldg(pl + (int64_t)p * rows + row));
  L = warp_max(L);
  float acc[Sh::kVpl * E];
#pragma unroll
  for (int i = 0; i < Sh::kVpl * E; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (L != -INFINITY) {
    for (int p0 = 0; p0 < num_splits; p0 += Sh::kGroups * Sh::kInFlight) {
      float w[Sh::kInFlight];
      uint4 v[Sh::kInFlight][Sh::kVpl];
#pragma unroll
      for (int i = 0; i < Sh::kInFlight; ++i) {
        const int p = p0 + g + i * Sh::kGroups;
        const float lp = p < num_splits ? __ldg(pl + (int64_t)p * rows + row) : -INFINITY;
        w[i] = lp == -INFINITY ? 0.f : __expf(lp - L);
        const uint4 *src = reinterpret_cast<const uint4 *>(po + ((int64_t)p * rows + row) * D);
#pragma unroll
        for (int j = 0; j < Sh::kVpl; ++j)
          v[i][j] = w[i] > 0.f ? __ldg(src + gl + j * Sh::kLanes) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < Sh::kInFlight; ++i) {
        wsum += w[i];
#pragma unroll
        for (int j = 0; j < Sh::kVpl; ++j) accum<T>(acc + j * E, v[i][j], w[i]);
      }
    }
  }
#pragma unroll
  for (int o = Sh::kLanes; o < 32; o <<= 1) {                // the groups' partial sums meet
    wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
#pragma unroll
    for (int i = 0; i < Sh::kVpl * E; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  }
  if (g != 0) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int i = 0; i < Sh::kVpl * E; ++i) acc[i] *= inv;
  uint4 *dst = reinterpret_cast<uint4 *>(out + row * D);
#pragma unroll
  for (int v = 0; v < Sh::kVpl; ++v) dst[gl + v * Sh::kLanes] = pack<T>(acc + v * E);
  if (out_lse != nullptr && gl == 0) out_lse[row] = (wsum > 0.f) ? L + logf(wsum) : -INFINITY;
}

// Below this many rows the warp-per-row kernel is used.
constexpr int64_t kRowWarpMaxRows = 32768;

// Launched as a programmatic dependent of the kernel before it in the stream
// (normally the split-KV attention, which lets it start during its tail): the
// kernels wait for it with pdl_wait() before they read the partials.
template <typename K, typename... Args>
cudaError_t launch_dependent(K kernel, int64_t grid, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename T, int D>
cudaError_t run(const void *po, const float *pl, int32_t P, int64_t rows, void *out, float *ol,
                cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const T *p = static_cast<const T *>(po);
  T *o = static_cast<T *>(out);
  if (rows < kRowWarpMaxRows)
    return launch_dependent(lse_combine_rowwarp_kernel<T, D>, ceil_div(rows, kThreads / 32), st, p, pl, P, rows, o, ol);
  using Sh = CombineShape<T, D>;
  const int64_t rows_per_block = (kThreads / 32) * Sh::kRowsPerWarp;
  return launch_dependent(lse_combine_kernel<T, D>, ceil_div(rows, rows_per_block), st, p, pl, P, rows, o, ol);
}

}  // namespace

cudaError_t launch_lse_combine(const void *po, const float *pl, int32_t num_splits,
                               int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                               int32_t dtype, void *out, float *out_lse, cudaStream_t st) {
  const int64_t rows = num_tokens * num_heads;
  if (dtype == SWA_DTYPE_BF16) {
    switch (head_dim) {
      case 64: return run<__nv_bfloat16, 64>(po, pl, num_splits, rows, out, out_lse, st);
      case 128: return run<__nv_bfloat16, 128>(po, pl, num_splits, rows, out, out_lse, st);
      case 256: return run<__nv_bfloat16, 256>(po, pl, num_splits, rows, out, out_lse, st);
    }
  } else {
    switch (head_dim) {
      case 64: return run<float, 64>(po, pl, num_splits, rows, out, out_lse, st);
      case 128: return run<float, 128>(po, pl, num_splits, rows, out, out_lse, st);
      case 256: return run<float, 256>(po, pl, num_splits, rows, out, out_lse, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace swa
