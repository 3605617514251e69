// Deterministic dK: a stable counting sort of the valid slots by key and a
// fixed-order segment sum of the per-slot dK rows.
//
// fp32 atomics make d_index_k run-to-run nondeterministic (cudnn-frontend #549
// "restore range_constexpr ...", numerics: dK uses fp32 atomicAdd and differs
// between reruns by ~1e-7; #707 makes the same point for red.global.add).
// Here the slots are first sorted by key:
//   sort:    for every key s, the slots (r, j) selecting it, in ascending
//            (r, j) order, from per-chunk histograms and a scan (no position
//            atomics, so the order is fixed);
// then the gemm kernel stores each slot's dK row in u, and
//   segsum:  dK[s] = sum of the key's u rows, in that order.
// Two layouts of u.  Position mode (a row's ids, dI and positions fit the
// gemm kernel's row stage): the sort gives each slot its position, the gemm
// kernel stores the slot's row there, so every key's rows are contiguous and
// the segment sum streams them.  Slot mode (longer rows): the gemm kernel
// stores slot r*L + j at row r*L + j, the sort lists the slots in key order,
// and the segment sum reads the rows through that list.
// The result is bitwise identical run to run and overwrites dK.
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace ibwd {
namespace {

constexpr int RB = kSortRows;  // query rows per sort chunk (chunks never straddle a batch)

__device__ __forceinline__ bool slot_key(const GemmArgs& a, long long r, int j, int& key) {
  if (a.idx) {
    const unsigned off = a.ids_global ? (unsigned)((int)r / a.S_q) * (unsigned)a.S_k : 0u;  // rows < 2^31
    key = (int)((unsigned)a.idx[r * a.L + j] - off);
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
// chunks (in place), and the key's total into key_start.  A block takes 32
// keys; its 32 warps split the batch's chunks into 32 contiguous segments
// (lane = key, so every access is a coalesced 128-byte row piece): segment
// sums, a scan over the segments, then the prefixes within each segment.
__global__ void __launch_bounds__(1024) colscan_kernel(const GemmArgs a, int* __restrict__ hist,
                                                      int* __restrict__ key_start) {
  __shared__ int seg[32][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int kpb = (a.S_k + 31) / 32;  // key blocks per batch
  const int b = (int)(blockIdx.x / kpb);
  const int s = (int)(blockIdx.x % kpb) * 32 + lane;
  const bool on = s < a.S_k;
  const int cpb = (a.S_q + RB - 1) / RB;
  const int per = (cpb + 31) / 32;
  const int c0 = min(cpb, w * per), c1 = min(cpb, c0 + per);
  int* col = hist + (long long)b * cpb * a.S_k + s;
  int sum = 0;
  if (on)
    for (int c = c0; c < c1; ++c) sum += col[(long long)c * a.S_k];
  seg[w][lane] = sum;
  __syncthreads();
  if (w == 0) {
    int run = 0;
    for (int k = 0; k < 32; ++k) {
      const int v = seg[k][lane];
      seg[k][lane] = run;
      run += v;
    }
    if (on) key_start[(long long)b * a.S_k + s] = run;
  }
  __syncthreads();
  if (on) {
    int run = seg[w][lane];
    for (int c = c0; c < c1; ++c) {
      int* h = col + (long long)c * a.S_k;
      const int v = *h;
      *h = run;
      run += v;
    }
  }
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

// One warp per chunk ranks its slots in ascending (r, j) order: lanes that
// hold the same key in one 32-slot step take consecutive positions by lane.
// Each row's ids are read 256 slots at a time into registers, one block
// ahead.  A step first tests for equal keys among its lanes (each lane tags
// its key in shared memory and reads the tag back): without duplicates every
// lane takes the key's cursor directly; with them the lanes rank themselves
// with a match.
// order: position mode, order[slot] = position; slot mode, order[position] = slot.
__global__ void __launch_bounds__(32) place_kernel(const GemmArgs a, const int* __restrict__ hist,
                                                   const int* __restrict__ key_start, int* __restrict__ order,
                                                   int position_mode) {
  extern __shared__ int cursor[];  // [S_k] cursors, then [S_k] one-byte tags
  unsigned char* tag = reinterpret_cast<unsigned char*>(cursor + a.S_k);
  const int cpb = (a.S_q + RB - 1) / RB;
  const long long chunk = blockIdx.x;
  const int b = (int)(chunk / cpb);
  const int t0 = (int)(chunk % cpb) * RB;
  const int lane = threadIdx.x;
  {
    const int* ks = key_start + (long long)b * a.S_k;
    const int* hs = hist + chunk * a.S_k;
    int s = lane;
    for (; s + 7 * 32 < a.S_k; s += 8 * 32) {
      int x[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = __ldg(ks + s + k * 32) + __ldg(hs + s + k * 32);
#pragma unroll
      for (int k = 0; k < 8; ++k) cursor[s + k * 32] = x[k];
    }
    for (; s < a.S_k; s += 32) cursor[s] = __ldg(ks + s) + __ldg(hs + s);
  }
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int t1 = min(a.S_q, t0 + RB);
  constexpr int NB = 8;  // 32-slot steps per register block
  // key of slot j of row r, or -1 when the slot is padding
  auto load_key = [&](long long r, int t, int j) -> int {
    const int lim = a.idx ? a.L : min(a.L, t + 1);
    if (j >= lim) return -1;
    if (!a.idx) return j;
    const unsigned off = a.ids_global ? (unsigned)((int)r / a.S_q) * (unsigned)a.S_k : 0u;  // rows < 2^31
    const int k = (int)((unsigned)__ldg(a.idx + r * a.L + j) - off);
    return (unsigned)k < (unsigned)a.S_k ? k : -1;
  };
  for (int t = t0; t < t1; ++t) {
    const long long r = (long long)b * a.S_q + t;
    const int lim = a.idx ? a.L : min(a.L, t + 1);
    int cur[NB], nxt[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) cur[k] = load_key(r, t, k * 32 + lane);
    for (int j0 = 0; j0 < lim; j0 += NB * 32) {
#pragma unroll
      for (int k = 0; k < NB; ++k) nxt[k] = load_key(r, t, j0 + NB * 32 + k * 32 + lane);
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        const int key = cur[k];
        const bool v = key >= 0;
        const int slot = (int)(r * a.L + j0 + k * 32 + lane);
        if (v) tag[key] = (unsigned char)lane;
        __syncwarp();
        const bool dup = __any_sync(0xffffffffu, v && tag[key] != lane);
        if (!dup) {
          if (v) {
            const int base = cursor[key];
            if (position_mode)
              order[slot] = base;
            else
              order[base] = slot;
            cursor[key] = base + 1;
          }
        } else {
          const unsigned grp = __match_any_sync(0xffffffffu, v ? key : -1 - lane);
          int base = 0;
          if (v) base = cursor[key];
          __syncwarp();
          if (v) {
            const int at = base + __popc(grp & lt);
            if (position_mode)
              order[slot] = at;
            else
              order[at] = slot;
            if ((grp & lt) == 0) cursor[key] = base + __popc(grp);
          }
        }
        __syncwarp();
      }
#pragma unroll
      for (int k = 0; k < NB; ++k) cur[k] = nxt[k];
    }
  }
}

// One block of eight warps per key: dK[key] = sum of the key's u rows, which
// the gemm kernel stored contiguously in position order.  Warp w sums rows
// w, w + 8, w + 16, ... of the segment in order (the block reads eight
// consecutive rows per step, four steps in flight), then the eight partial
// sums are added in warp order: a fixed order, so dK is bitwise reproducible.
constexpr int SEG_WARPS = 8;
// perm: slot mode, the key-order slot list (u row of position p is perm[p]);
// position mode, nullptr (u row p).
__global__ void __launch_bounds__(SEG_WARPS * 32) segsum_kernel(const GemmArgs a, const float* __restrict__ u,
                                                               const int* __restrict__ key_start,
                                                               const int* __restrict__ perm) {
  __shared__ float4 part[SEG_WARPS][32];
  const long long gk = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int beg = key_start[gk], end = key_start[gk + 1];
  const int d = lane * 4;
  const bool on = d < a.D;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int NF = 4;  // steps in flight per warp
  for (int p0 = beg + w; p0 < end; p0 += NF * SEG_WARPS) {
    int sl[NF];  // the steps' slots, whose dK rows are u[slot]
#pragma unroll
    for (int k = 0; k < NF; ++k) {
      const int pr = p0 + k * SEG_WARPS;
      sl[k] = pr < end ? (perm ? __ldg(perm + pr) : pr) : 0;
    }
    float4 v[NF];
#pragma unroll
    for (int k = 0; k < NF; ++k) {
      const int pr = p0 + k * SEG_WARPS;
      v[k] = (on && pr < end) ? __ldcs(reinterpret_cast<const float4*>(u + (long long)sl[k] * a.D + d))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < NF; ++k) {
      if (p0 + k * SEG_WARPS < end) {
        acc.x += v[k].x;
        acc.y += v[k].y;
        acc.z += v[k].z;
        acc.w += v[k].w;
      }
    }
  }
  part[w][lane] = acc;
  __syncthreads();
  if (w == 0 && on) {
    float4 t = part[0][lane];
#pragma unroll
    for (int k = 1; k < SEG_WARPS; ++k) {
      const float4 x = part[k][lane];
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
    *reinterpret_cast<float4*>(a.dk + gk * a.D + d) = t;
  }
}

}  // namespace

cudaError_t launch_det_sort(const GemmArgs& a, const WsLayout& lay, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  int* hist = reinterpret_cast<int*>(ws + lay.hist);
  int* key_start = reinterpret_cast<int*>(ws + lay.key_start);
  int* order = reinterpret_cast<int*>(ws + lay.order);
  const size_t sh = (size_t)a.S_k * sizeof(int);       // histogram counters
  const size_t sh_place = sh + (size_t)a.S_k;              // cursors and one-byte tags
  static std::atomic<bool> attr_set[64];  // per device; setting the attribute twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (sh_place > 48 * 1024 && dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  hist_kernel<<<(unsigned)lay.nchunks, 256, sh, st>>>(a, hist);
  const long long nk = (long long)a.B * a.S_k;
  colscan_kernel<<<(unsigned)(a.B * ((a.S_k + 31) / 32)), 1024, 0, st>>>(a, hist, key_start);
  keyscan_kernel<<<1, 1024, 0, st>>>(key_start, nk);
  place_kernel<<<(unsigned)lay.nchunks, 32, sh_place, st>>>(a, hist, key_start, order, det_position_mode(a) ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_det_segsum(const GemmArgs& a, const WsLayout& lay, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  const float* u = reinterpret_cast<const float*>(ws + lay.u);
  const int* key_start = reinterpret_cast<const int*>(ws + lay.key_start);
  const int* perm = det_position_mode(a) ? nullptr : reinterpret_cast<const int*>(ws + lay.order);
  const long long nk = (long long)a.B * a.S_k;
  segsum_kernel<<<(unsigned)nk, SEG_WARPS * 32, 0, st>>>(a, u, key_start, perm);
  return cudaGetLastError();
}

}  // namespace ibwd
