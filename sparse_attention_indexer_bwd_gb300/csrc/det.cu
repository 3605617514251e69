// Deterministic dK: a stable counting sort of the blocks' entries by key and
// a fixed-order segment sum of the per-entry dK rows.
//
// fp32 atomics make d_index_k run-to-run nondeterministic (cudnn-frontend #549
// "restore range_constexpr ...", numerics: dK uses fp32 atomicAdd and differs
// between reruns by ~1e-7; #707 makes the same point for red.global.add).
// The gemm kernel works on blocks of four query rows and gives one dK row per
// (block, key) entry (the four rows' contributions already summed by the
// tensor core).  Here every entry gets a position such that each key's
// entries are contiguous and in ascending block order; the gemm kernel stores
// the entry's row there, in fp16 under a power-of-two scale bounded from the
// block's largest |q| and dz scale (no row can reach the fp16 limit; the
// rounding is 2^-12 of the row's own values), with its restoring factor, and
//   segsum:  dK[s] = sum of the key's rows times their factors, in that order.
// fp16 rows halve the traffic of the mode's HBM-bound part (the rows are
// written once and read once).
// Sparse: per chunk of kSortBlocks blocks, per-key counts (a key appears at
// most once per block; the union pass counts them as it writes the records),
// an exclusive scan over the chunks and over the keys (no position atomics,
// so the order is fixed), then the positions, written into the tile records.
// Dense: block j of a batch holds keys [0, 4j + Rb), so the positions have
// a closed form (the gemm kernel computes them) and only the CSR offsets are
// filled here.
// The result is bitwise identical run to run and overwrites dK.
#include <algorithm>
#include <atomic>

#include "kcommon.cuh"

namespace ibwd {
namespace {

constexpr int CB = kSortBlocks;  // blocks per sort chunk (chunks never straddle a batch)
constexpr int REC_KEY = 0, REC_POS = 2560;

struct DetP {
  char* rec;
  const int4* binfo;
  long long nblocks;
  int S_k, nbpb, tcap, rstride;
};

__device__ __forceinline__ int* rec_field(const DetP& d, long long b, int e, int off) {
  return reinterpret_cast<int*>(d.rec + (b * d.tcap + (e >> 7)) * d.rstride + off) + (e & 127);
}

// Exclusive scan of the per-key totals into CSR offsets, by one CTA of 1024
// threads (the totals were written by other CTAs: read past L1).
__device__ __forceinline__ void keyscan(int* __restrict__ key_start, long long n) {
  __shared__ int part[1024];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (long long base = 0; base < n; base += 1024) {
    const long long i = base + threadIdx.x;
    const int v = i < n ? __ldcg(key_start + i) : 0;
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

// For each (batch, key): exclusive prefix of the counts over the batch's
// chunks (in place), and the key's total into key_start.  A block takes 32
// keys; its 32 warps split the batch's chunks into 32 contiguous segments
// (lane = key, so every access is a coalesced 128-byte row piece): segment
// sums, a scan over the segments, then the prefixes within each segment.
// The counts come from the union pass (one per block entry).  The last CTA
// to finish turns every batch's key totals into CSR offsets.
__global__ void __launch_bounds__(1024) colscan_kernel(int* __restrict__ hist, int* __restrict__ key_start, int S_k,
                                                      int cpb, int B, unsigned* __restrict__ done) {
  __shared__ int seg[32][33];
  __shared__ int s_last;
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int kpb = (S_k + 31) / 32;  // key blocks per batch
  const int b = (int)(blockIdx.x / kpb);
  const int s = (int)(blockIdx.x % kpb) * 32 + lane;
  const bool on = s < S_k;
  const int per = (cpb + 31) / 32;
  const int c0 = min(cpb, w * per), c1 = min(cpb, c0 + per);
  int* col = hist + (long long)b * cpb * S_k + s;
  int sum = 0;
  if (on)
    for (int c = c0; c < c1; ++c) sum += col[(long long)c * S_k];
  seg[w][lane] = sum;
  __syncthreads();
  if (w == 0) {
    int run = 0;
    for (int k = 0; k < 32; ++k) {
      const int v = seg[k][lane];
      seg[k][lane] = run;
      run += v;
    }
    if (on) key_start[(long long)b * S_k + s] = run;
  }
  __syncthreads();
  if (on) {
    int run = seg[w][lane];
    for (int c = c0; c < c1; ++c) {
      int* h = col + (long long)c * S_k;
      const int v = *h;
      *h = run;
      run += v;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  keyscan(key_start, (long long)B * S_k);
}

// Positions of a chunk's entries: each key's cursor starts at its CSR offset
// plus the count of the batch's earlier chunks; the chunk's blocks take their
// positions in block order, all entries of a block at once (its keys are
// distinct).
__global__ void __launch_bounds__(256) place_kernel(const DetP d, const int* __restrict__ hist,
                                                   const int* __restrict__ key_start) {
  extern __shared__ int cursor[];
  griddep_launch_dependents();
  griddep_wait();  // the offsets come from the column scan
  const int cpb = (d.nbpb + CB - 1) / CB;
  const long long chunk = blockIdx.x;
  const int bb = (int)(chunk / cpb), j0 = (int)(chunk % cpb) * CB;
  const int* ks = key_start + (long long)bb * d.S_k;
  const int* hs = hist + chunk * d.S_k;
  for (int s = threadIdx.x; s < d.S_k; s += blockDim.x) cursor[s] = __ldg(ks + s) + __ldg(hs + s);
  __syncthreads();
  for (int jb = j0; jb < min(d.nbpb, j0 + CB); ++jb) {
    const long long b = (long long)bb * d.nbpb + jb;
    const int U = __ldg(&d.binfo[b].z);
    for (int e = threadIdx.x; e < U; e += blockDim.x) {
      const int key = *rec_field(d, b, e, REC_KEY);
      const int pos = cursor[key];
      cursor[key] = pos + 1;
      *rec_field(d, b, e, REC_POS) = pos;
    }
    __syncthreads();
  }
}

// Dense CSR offsets: key s of a batch lies in blocks floor(s/4) .. nbpb-1, so
// the keys before it hold s*nbpb - sum_{s'<s} floor(s'/4) entries.
__global__ void dense_keystart_kernel(int* __restrict__ key_start, int B, int S, int nbpb, long long per_batch) {
  const long long n = (long long)B * S;
  griddep_launch_dependents();
  griddep_wait();
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x <= n; x += (long long)gridDim.x * blockDim.x) {
    const long long bb = x / S, s = x % S;
    const long long a = s >> 2, c = s & 3;
    key_start[x] = (int)(bb * per_batch + s * nbpb - (2 * a * (a - 1) + c * a));
  }
}

// One block of eight warps per key: dK[key] = sum of the key's u rows, which
// the gemm kernel stored contiguously in position order as fp16 rows, each
// with its restoring factor.  Warp w sums rows w, w + 8, w + 16, ... of the
// segment in order (the block reads eight consecutive rows per step, NF steps
// in flight), then the eight partial sums are added in warp order: a fixed
// order, so dK is bitwise reproducible.
constexpr int SEG_WARPS = 8;
__global__ void __launch_bounds__(SEG_WARPS * 32) segsum_kernel(const char* __restrict__ u,
                                                               const int* __restrict__ key_start,
                                                               float* __restrict__ dk, int D) {
  __shared__ float4 part[SEG_WARPS][32];
  griddep_wait();  // the u rows come from the gemm kernel
  const long long gk = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int beg = key_start[gk], end = key_start[gk + 1];
  const int d = lane * 4;
  const bool on = d < D;
  const int rb = u_row_bytes(D), fsec = rb - 32;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int NF = 8;  // steps in flight per warp
  for (int p0 = beg + w; p0 < end; p0 += NF * SEG_WARPS) {
    uint2 v[NF];
    float f[NF];
#pragma unroll
    for (int k = 0; k < NF; ++k) {
      const int pr = p0 + k * SEG_WARPS;
      const bool in = pr < end;
      const char* row = u + (long long)pr * rb;
      v[k] = (on && in) ? __ldcs(reinterpret_cast<const uint2*>(row + 2 * d)) : make_uint2(0u, 0u);
      f[k] = in ? __ldcs(reinterpret_cast<const float*>(row + fsec)) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < NF; ++k) {
      if (p0 + k * SEG_WARPS < end) {
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&v[k].x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&v[k].y));
        acc.x += lo.x * f[k];
        acc.y += lo.y * f[k];
        acc.z += hi.x * f[k];
        acc.w += hi.y * f[k];
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
    *reinterpret_cast<float4*>(dk + gk * D + d) = t;
  }
}

std::atomic<int> g_attr_place[64];

bool raise_smem(const void* fn, size_t bytes, std::atomic<int>* done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire) >= (int)bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) return false;
  if (dev >= 0 && dev < 64) done[dev].store((int)bytes, std::memory_order_release);
  return true;
}

}  // namespace

cudaError_t launch_det_sort(const GemmArgs& a, const WsLayout& lay, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  int* key_start = reinterpret_cast<int*>(ws + lay.key_start);
  if (!a.idx) {
    const long long n = (long long)a.B * a.S_k + 1;
    const int blocks = (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, 4LL * a.num_sms));
    return launch_ex(dense_keystart_kernel, (unsigned)blocks, 256u, 0, st, true, key_start, a.B, a.S_k, lay.nbpb,
                     lay.entries_cap / a.B);
  }
  DetP d{};
  d.rec = ws + lay.rec;
  d.binfo = reinterpret_cast<const int4*>(ws + lay.binfo);
  d.nblocks = lay.nblocks;
  d.S_k = a.S_k;
  d.nbpb = lay.nbpb;
  d.tcap = lay.tcap;
  d.rstride = lay.rstride;
  int* hist = reinterpret_cast<int*>(ws + lay.hist);
  const size_t sh = (size_t)a.S_k * sizeof(int);  // per-key counters or cursors
  if (!raise_smem((const void*)place_kernel, sh, g_attr_place)) return cudaErrorInvalidValue;
  const int cpb = (lay.nbpb + CB - 1) / CB;
  unsigned* done = reinterpret_cast<unsigned*>(ws + lay.sched) + kSchedDetScan;  // zeroed by the k copy
  cudaError_t e = launch_ex(colscan_kernel, (unsigned)(a.B * ((a.S_k + 31) / 32)), 1024u, 0, st, true, hist,
                            key_start, a.S_k, cpb, a.B, done);
  if (e != cudaSuccess) return e;
  return launch_ex(place_kernel, (unsigned)lay.nchunks, 256u, sh, st, true, static_cast<const DetP>(d),
                   static_cast<const int*>(hist), static_cast<const int*>(key_start));
}

cudaError_t launch_det_segsum(const GemmArgs& a, const WsLayout& lay, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  const char* u = ws + lay.u;
  const int* key_start = reinterpret_cast<const int*>(ws + lay.key_start);
  const long long nk = (long long)a.B * a.S_k;
  return launch_ex(segsum_kernel, (unsigned)nk, (unsigned)(SEG_WARPS * 32), 0, st, true, u, key_start, a.dk, a.D);
}

}  // namespace ibwd
