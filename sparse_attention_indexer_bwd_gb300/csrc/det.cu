// Deterministic dK: a stable counting sort of the valid slots by key and a
// fixed-order segment sum of the per-slot dK rows.
//
// fp32 atomics make d_index_k run-to-run nondeterministic (cudnn-frontend #549
// "restore range_constexpr ...", numerics: dK uses fp32 atomicAdd and differs
// between reruns by ~1e-7; #707 makes the same point for red.global.add).
// Here the gemm kernel stores each slot's dK row u[r*L + j] instead, and
//   sort:    for every key s, the slots (r, j) selecting it, in ascending
//            (r, j) order, from per-chunk histograms and a scan (no position
//            atomics, so the order is fixed);
//   segsum:  dK[s] = sum over that list, in that order, of u rows.
// The result is bitwise identical run to run and overwrites dK.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace ibwd {
namespace {

constexpr int RB = 16;  // query rows per sort chunk (chunks never straddle a batch)

__device__ __forceinline__ bool slot_key(const GemmArgs& a, long long r, int j, int& key) {
  if (a.idx) {
    key = a.idx[r * a.L + j];
    return (unsigned)key < (unsigned)a.S_k;
  }
  key = j;
  return j <= (int)(r % a.S_q);
}

// Counts, per chunk of RB rows, how many valid slots select each key.
__global__ void __launch_bounds__(256) hist_kernel(const GemmArgs a, int* __restrict__ hist) {
  extern __shared__ int sh[];
  const int cpb = (a.S_q + RB - 1) / RB;  // chunks per batch
  const long long chunk = blockIdx.x;
  const int b = (int)(chunk / cpb);
  const int t0 = (int)(chunk % cpb) * RB;
  for (int s = threadIdx.x; s < a.S_k; s += blockDim.x) sh[s] = 0;
  __syncthreads();
  const int t1 = min(a.S_q, t0 + RB);
  for (int t = t0; t < t1; ++t) {
    const long long r = (long long)b * a.S_q + t;
    for (int j = threadIdx.x; j < a.L; j += blockDim.x) {
      int key;
      if (slot_key(a, r, j, key)) atomicAdd(&sh[key], 1);
    }
  }
  __syncthreads();
  for (int s = threadIdx.x; s < a.S_k; s += blockDim.x) hist[chunk * a.S_k + s] = sh[s];
}

// For each (batch, key): exclusive prefix of the counts over the batch's
// chunks (in place), and the key's total into key_start.
__global__ void colscan_kernel(const GemmArgs a, int* __restrict__ hist, int* __restrict__ key_start) {
  const long long gk = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (gk >= (long long)a.B * a.S_k) return;
  const int b = (int)(gk / a.S_k), s = (int)(gk % a.S_k);
  const int cpb = (a.S_q + RB - 1) / RB;
  int run = 0;
  for (int c = 0; c < cpb; ++c) {
    int* h = hist + ((long long)b * cpb + c) * a.S_k + s;
    const int v = *h;
    *h = run;
    run += v;
  }
  key_start[gk] = run;
}

// Exclusive scan of the per-key totals into CSR offsets (one block).
__global__ void __launch_bounds__(1024) keyscan_kernel(int* __restrict__ key_start, long long n) {
  __shared__ int part[1024];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (long long base = 0; base < n; base += 1024) {
    const long long i = base + threadIdx.x;
    const int v = i < n ? key_start[i] : 0;
    part[threadIdx.x] = v;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
      const int add = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
      __syncthreads();
      part[threadIdx.x] += add;
      __syncthreads();
    }
    const int excl = part[threadIdx.x] - v + carry;
    if (i < n) key_start[i] = excl;
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) key_start[n] = carry;
}

// One warp per chunk places its slots in ascending (r, j) order: lanes that
// hold the same key in one 32-slot step take consecutive positions by lane.
__global__ void __launch_bounds__(32) place_kernel(const GemmArgs a, const int* __restrict__ hist,
                                                   const int* __restrict__ key_start, int* __restrict__ perm) {
  extern __shared__ int cursor[];
  const int cpb = (a.S_q + RB - 1) / RB;
  const long long chunk = blockIdx.x;
  const int b = (int)(chunk / cpb);
  const int t0 = (int)(chunk % cpb) * RB;
  const int lane = threadIdx.x;
  for (int s = lane; s < a.S_k; s += 32)
    cursor[s] = key_start[(long long)b * a.S_k + s] + hist[chunk * a.S_k + s];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int t1 = min(a.S_q, t0 + RB);
  for (int t = t0; t < t1; ++t) {
    const long long r = (long long)b * a.S_q + t;
    const int lim = a.idx ? a.L : min(a.L, t + 1);
    for (int j0 = 0; j0 < lim; j0 += 32) {
      const int j = j0 + lane;
      int key = 0;
      const bool v = j < lim && slot_key(a, r, j, key);
      const unsigned grp = __match_any_sync(0xffffffffu, v ? key : -1 - lane);
      int base = 0;
      if (v) base = cursor[key];
      __syncwarp();
      if (v) {
        perm[base + __popc(grp & lt)] = (int)(r * a.L + j);
        if ((grp & lt) == 0) cursor[key] = base + __popc(grp);
      }
      __syncwarp();
    }
  }
}

// One warp per key: dK[key] = sum of u rows over the key's CSR segment, in
// segment order.
__global__ void __launch_bounds__(256) segsum_kernel(const GemmArgs a, const float* __restrict__ u,
                                                     const int* __restrict__ key_start,
                                                     const int* __restrict__ perm) {
  const long long gk = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gk >= (long long)a.B * a.S_k) return;
  const int beg = key_start[gk], end = key_start[gk + 1];
  const int d = lane * 4;
  const bool on = d < a.D;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int p = beg;
  for (; p + 4 <= end; p += 4) {
    const int i0 = __ldg(perm + p), i1 = __ldg(perm + p + 1), i2 = __ldg(perm + p + 2), i3 = __ldg(perm + p + 3);
    if (on) {
      const float4 v0 = __ldcs(reinterpret_cast<const float4*>(u + (long long)i0 * a.D + d));
      const float4 v1 = __ldcs(reinterpret_cast<const float4*>(u + (long long)i1 * a.D + d));
      const float4 v2 = __ldcs(reinterpret_cast<const float4*>(u + (long long)i2 * a.D + d));
      const float4 v3 = __ldcs(reinterpret_cast<const float4*>(u + (long long)i3 * a.D + d));
      acc.x += v0.x; acc.y += v0.y; acc.z += v0.z; acc.w += v0.w;
      acc.x += v1.x; acc.y += v1.y; acc.z += v1.z; acc.w += v1.w;
      acc.x += v2.x; acc.y += v2.y; acc.z += v2.z; acc.w += v2.w;
      acc.x += v3.x; acc.y += v3.y; acc.z += v3.z; acc.w += v3.w;
    }
  }
  for (; p < end; ++p) {
    const int i0 = __ldg(perm + p);
    if (on) {
      const float4 v0 = __ldcs(reinterpret_cast<const float4*>(u + (long long)i0 * a.D + d));
      acc.x += v0.x; acc.y += v0.y; acc.z += v0.z; acc.w += v0.w;
    }
  }
  if (on) *reinterpret_cast<float4*>(a.dk + gk * a.D + d) = acc;
}

}  // namespace

cudaError_t launch_det_sort(const GemmArgs& a, const WsLayout& lay, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  int* hist = reinterpret_cast<int*>(ws + lay.hist);
  int* key_start = reinterpret_cast<int*>(ws + lay.key_start);
  int* perm = reinterpret_cast<int*>(ws + lay.perm);
  const size_t sh = (size_t)a.S_k * sizeof(int);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (sh > 48 * 1024 && dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  hist_kernel<<<(unsigned)lay.nchunks, 256, sh, st>>>(a, hist);
  const long long nk = (long long)a.B * a.S_k;
  colscan_kernel<<<(unsigned)((nk + 255) / 256), 256, 0, st>>>(a, hist, key_start);
  keyscan_kernel<<<1, 1024, 0, st>>>(key_start, nk);
  place_kernel<<<(unsigned)lay.nchunks, 32, sh, st>>>(a, hist, key_start, perm);
  return cudaGetLastError();
}

cudaError_t launch_det_segsum(const GemmArgs& a, const WsLayout& lay, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  const float* u = reinterpret_cast<const float*>(ws + lay.u);
  const int* key_start = reinterpret_cast<const int*>(ws + lay.key_start);
  const int* perm = reinterpret_cast<const int*>(ws + lay.perm);
  const long long nk = (long long)a.B * a.S_k;
  segsum_kernel<<<(unsigned)((nk * 32 + 255) / 256), 256, 0, st>>>(a, u, key_start, perm);
  return cudaGetLastError();
}

}  // namespace ibwd
