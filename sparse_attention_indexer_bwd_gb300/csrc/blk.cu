// The union pass, the k conversion and the host side of the blocked gemm
// stage: workspace layout and the launch sequence (the gemm kernel itself is
// in blk_pipe.cuh).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdlib>
#include <cstring>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "blk.h"

namespace ibwd {
using namespace blk;
namespace {


// ------------------------------------------------------------ union pass --
constexpr int UT = 256;        // threads: warps r and r + 4 handle row r of the block
constexpr int NBUCKET = 1024;  // tile-count buckets of the block order

struct UParams {
  const int32_t* idx;  // [rows, L]
  const float* dI;     // [rows, L]
  const float* w;      // [rows, H]
  char* rec;           // tile records
  int4* binfo;         // per block {tiles, c, entries, 0}
  int* border;         // blocks in descending tile count (written by the last CTA)
  unsigned* done;      // CTA counter, zeroed by the k conversion kernel
  long long nblocks;
  int S_q, S_k, H, L, nbpb, tcap, rstride, ids_global;
  int* hist;   // deterministic mode: per (sort chunk, key) counts of the chunk's blocks holding the key, or nullptr
  int cpb;     // deterministic mode: sort chunks per batch
  int W;       // key window per pass (multiple of 1024)
  int dcap;    // per-row capacity of the dedup arrays: min(L, W)
  int staged;    // the block's id rows are copied into shared memory (Lp = L rounded up to 4)
  int staged_dI;  // and its dI rows after them (read once each: not for long rows, where shared memory sets the occupancy)
  const unsigned* select;  // if set: the pass runs only when *select == 0 (1 selects the per-row kernel)
};

// Exclusive prefix of the popcounts of n words (n a multiple of 32), by one
// warp; returns the total.
__device__ __forceinline__ int warp_popc_prefix(const uint32_t* bm, int* pf, int n) {
  const int lane = threadIdx.x & 31;
  const int per = n >> 5;
  const uint32_t* src = bm + lane * per;
  int sum = 0;
  for (int i = 0; i < per; ++i) sum += __popc(src[i]);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;
  int* dst = pf + lane * per;
  for (int i = 0; i < per; ++i) {
    dst[i] = run;
    run += __popc(src[i]);
  }
  return __shfl_sync(FULL, incl, 31);
}

// Copies the block's rows of a [rows, L] array into shared memory rows of Lp
// elements (cp.async: 16-byte pieces when the rows are 16-byte aligned, else
// 4-byte ones), all in flight at once; the caller waits.
__device__ __forceinline__ void stage_rows(uint32_t dst, const void* src_base, long long row0, int Rb, int L, int Lp) {
  const char* src = static_cast<const char*>(src_base) + row0 * L * 4;
  if ((L & 3) == 0) {
    const int per = L >> 2;  // 16-byte pieces per row
    for (int x = threadIdx.x; x < Rb * per; x += UT) {
      const int r = x / per, c = x - r * per;
      cp_async16(dst + (uint32_t)(r * Lp + 4 * c) * 4, src + ((long long)r * L + 4 * c) * 4, 16);
    }
  } else {
    for (int x = threadIdx.x; x < Rb * L; x += UT) {
      const int r = x / L, c = x - r * L;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst + (uint32_t)(r * Lp + c) * 4),
                   "l"(src + ((long long)r * L + c) * 4)
                   : "memory");
    }
  }
  cp_async_commit();
}

// One CTA per block.  Per window of W keys: a bitmap of each row's valid keys
// and of their union; popcount prefixes give every key its rank (row-local
// and union); each row's dI is summed per distinct key in slot order (rows
// with repeated ids: lanes holding the same key in one 32-slot step add their
// values in lane order, steps in slot order, so the sum is fixed; a step
// takes as many shuffle rounds as its largest group of equal keys); then the
// union's entries are written in ascending key order with the four rows'
// sums.  The largest |dis| * |w| of the block fixes its dz scale.  The last
// CTA to finish orders all blocks by descending tile count (a processing
// order for the gemm kernel; it affects no result).
__global__ void __launch_bounds__(UT, 4) union_kernel(const UParams p) {
  extern __shared__ __align__(16) uint32_t us[];
  const int WW = p.W >> 5;
  const int Lp = (p.L + 3) & ~3;
  uint32_t* bm = us;                                      // [5][WW]: rows 0-3, union
  int* pf = reinterpret_cast<int*>(us + 5 * WW);          // [5][WW]
  float* drow = reinterpret_cast<float*>(us + 10 * WW);   // [4][dcap]
  int* ids_s = reinterpret_cast<int*>(drow + R * p.dcap);  // staged: [4][Lp] ids, then [4][Lp] dI
  float* dI_s = reinterpret_cast<float*>(ids_s + R * Lp);
  constexpr int NW = UT / 32;
  __shared__ int s_cnt[5], s_kmin[NW], s_kmax[NW], s_dup[NW];
  __shared__ float s_wmax[R], s_dmax[NW][R];
  __shared__ int s_last;
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warp w: row w % 4, and of its slots the 32-slot steps of parity w / 4
  const int row = warp & 3, hlf = warp >> 2;
  const long long b = blockIdx.x;
  const int bb = (int)(b / p.nbpb), jb = (int)(b % p.nbpb);
  const int t0 = jb * R;
  const int Rb = min(R, p.S_q - t0);
  const long long row0 = (long long)bb * p.S_q + t0;
  const unsigned off = p.ids_global ? (unsigned)bb * (unsigned)p.S_k : 0u;  // rows < 2^31
  const bool own = row < Rb;
  // this warp's row: in shared memory when staged, else global
  const int32_t* ir = p.staged ? ids_s + row * Lp : p.idx + (own ? (row0 + row) * p.L : 0);
  const float* dr_in = p.staged_dI ? dI_s + row * Lp : p.dI + (own ? (row0 + row) * p.L : 0);
  if (p.staged) stage_rows(smem_u32(ids_s), p.idx, row0, Rb, p.L, Lp);

  float wmax = 0.f;  // over the row's heads
  if (own && hlf == 0) {
    for (int h = lane; h < p.H; h += 32) {
      const float a = fabsf(__ldg(p.w + (row0 + row) * p.H + h));
      wmax = fmaxf(wmax, a);
    }
    wmax = warp_max(wmax);
  }
  // dI is written by an earlier kernel (score-grad), the choice of gemm
  // kernel by the one before (its launch lets this one start early); the
  // dI copy then joins the ids copy in flight
  griddep_wait();
  const bool rows_path = p.select && __ldcg(p.select) != 0u;  // the per-row kernel serves this call
  if (p.staged) {
    if (!rows_path && p.staged_dI) stage_rows(smem_u32(dI_s), p.dI, row0, Rb, p.L, Lp);
    cp_async_wait_all();
    __syncthreads();
  }
  if (rows_path) return;
  // key range of the block's valid slots (one window covers every key when S_k <= W)
  int kmin = 0, kmax = p.S_k - 1;
  if (p.S_k > p.W) {
    kmin = INT_MAX;
    kmax = -1;
    if (own) {
      for (int j = lane + 32 * hlf; j < p.L; j += 64) {
        const int s = (int)((unsigned)ir[j] - off);
        if ((unsigned)s < (unsigned)p.S_k) {
          kmin = min(kmin, s);
          kmax = max(kmax, s);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(FULL, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(FULL, kmax, o));
      }
    }
    if (lane == 0) {
      s_kmin[warp] = kmin;
      s_kmax[warp] = kmax;
    }
  }
  if (lane == 0 && hlf == 0) s_wmax[row] = wmax;
  __syncthreads();
  if (p.S_k > p.W) {
    for (int x = 0; x < NW; ++x) {
      kmin = min(kmin, s_kmin[x]);
      kmax = max(kmax, s_kmax[x]);
    }
  }
  float dmax[R] = {0.f, 0.f, 0.f, 0.f};
  int base = 0;
  for (long long w0l = kmin; w0l <= kmax; w0l += p.W) {  // no pass when the block has no valid slot
    const int w0 = (int)w0l;
    for (int i = tid; i < 5 * WW; i += UT) bm[i] = 0u;
    __syncthreads();
    bool dup = false;
    if (own) {
      // four slots' atomics in flight at a time
      for (int j0 = lane + 32 * hlf; j0 < p.L; j0 += 4 * 64) {
        unsigned xs[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int j = j0 + 64 * t;
          xs[t] = 0xFFFFFFFFu;
          if (j < p.L) {
            const int s = (int)((unsigned)ir[j] - off);
            const unsigned x = (unsigned)(s - w0);
            if ((unsigned)s < (unsigned)p.S_k && x < (unsigned)p.W) xs[t] = x;
          }
        }
        uint32_t old[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          old[t] = xs[t] != 0xFFFFFFFFu ? atomicOr(&bm[row * WW + (xs[t] >> 5)], 1u << (xs[t] & 31)) : 0u;
#pragma unroll
        for (int t = 0; t < 4; ++t) dup |= xs[t] != 0xFFFFFFFFu && ((old[t] >> (xs[t] & 31)) & 1u);
      }
    }
    dup = __any_sync(FULL, dup);
    if (lane == 0) s_dup[warp] = dup;
    __syncthreads();
    // a key set twice in a row, by either of its warps
    dup = s_dup[row] | s_dup[row + 4];
    for (int i = tid; i < WW; i += UT) bm[4 * WW + i] = bm[i] | bm[WW + i] | bm[2 * WW + i] | bm[3 * WW + i];
    __syncthreads();
    for (int x = warp; x < 5; x += UT / 32) {
      const int n = warp_popc_prefix(bm + x * WW, pf + x * WW, WW);
      if (lane == 0) s_cnt[x] = n;
    }
    __syncthreads();
    // a row without repeated keys: each of its warps stores its own slots'
    // dI at their ranks; a row with repeats: its first warp alone adds the
    // row's values per key in slot order
    if (own && (!dup || hlf == 0)) {
      float* drr = drow + row * p.dcap;
      const uint32_t* bmr = bm + row * WW;
      const int* pfr = pf + row * WW;
      if (dup) {
        for (int i = lane; i < s_cnt[row]; i += 32) drr[i] = 0.f;
        __syncwarp();
      }
      // NBT steps at a time: their ids, ranks and dI (from global memory for
      // long rows) are all read before any is used, so the loads overlap;
      // the steps are then taken in order (a row with repeats sums in slot
      // order)
      constexpr int NBT = 4;
      const int jstep = dup ? 32 : 64;
      for (int j0 = dup ? 0 : 32 * hlf; j0 < p.L; j0 += NBT * jstep) {
        int rk[NBT];
        float vv[NBT];
#pragma unroll
        for (int t = 0; t < NBT; ++t) {
          const int j = j0 + t * jstep + lane;
          rk[t] = -1;
          vv[t] = 0.f;
          if (j < p.L) {
            const int s = (int)((unsigned)ir[j] - off);
            const unsigned x = (unsigned)(s - w0);
            if ((unsigned)s < (unsigned)p.S_k && x < (unsigned)p.W) {
              rk[t] = pfr[x >> 5] + __popc(bmr[x >> 5] & ((1u << (x & 31)) - 1u));
              vv[t] = p.staged_dI ? dr_in[j] : __ldg(dr_in + j);
            }
          }
        }
        if (!dup) {
#pragma unroll
          for (int t = 0; t < NBT; ++t)
            if (rk[t] >= 0) drr[rk[t]] = vv[t];
        } else {
          // per step, the lanes of each lane's group (same key) in lane
          // order: as many shuffle rounds as the step's largest group; the
          // steps' groups are independent, their additions into the sums
          // are made in step order
          unsigned grp[NBT];
#pragma unroll
          for (int t = 0; t < NBT; ++t) grp[t] = __match_any_sync(FULL, rk[t] >= 0 ? rk[t] : -1 - lane);
          int rounds = 0;
#pragma unroll
          for (int t = 0; t < NBT; ++t) rounds = max(rounds, __popc(grp[t]));
          rounds = (int)__reduce_max_sync(FULL, (unsigned)rounds);
          float sum[NBT];
          unsigned rest[NBT];
#pragma unroll
          for (int t = 0; t < NBT; ++t) {
            sum[t] = 0.f;
            rest[t] = grp[t];
          }
          for (int k = 0; k < rounds; ++k) {
#pragma unroll
            for (int t = 0; t < NBT; ++t) {
              const float y = __shfl_sync(FULL, vv[t], rest[t] ? __ffs(rest[t]) - 1 : lane);
              if (rest[t]) {
                sum[t] += y;
                rest[t] &= rest[t] - 1u;
              }
            }
          }
#pragma unroll
          for (int t = 0; t < NBT; ++t) {
            if (rk[t] >= 0 && (grp[t] & ((1u << lane) - 1u)) == 0u) drr[rk[t]] += sum[t];
            __syncwarp();
          }
        }
      }
    }
    __syncthreads();
    // the union's entries of this window, in ascending key order: a warp
    // takes one bitmap word at a time and lane l its bit l, so the set lanes
    // write consecutive entries; empty words (about half of them for causal
    // rows) are passed over at once
    // (every shared read of a word comes before its global stores, so the
    // reads overlap)
    for (int i = warp; i < WW; i += UT / 32) {
      const uint32_t m = bm[4 * WW + i];
      if (m == 0u) continue;  // warp-uniform: one word for all lanes
      const bool on = (m >> lane) & 1u;
      const uint32_t below = (1u << lane) - 1u;
      const int pu = pf[4 * WW + i];
      uint32_t mr[R];
      int pr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        mr[r] = bm[r * WW + i];
        pr[r] = pf[r * WW + i];
      }
      float d[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        d[r] = (on && ((mr[r] >> lane) & 1u)) ? drow[r * p.dcap + pr[r] + __popc(mr[r] & below)] : 0.f;
      if (!on) continue;
      const int ug = base + pu + __popc(m & below);
      char* rb = p.rec + ((long long)b * p.tcap + (ug >> 7)) * p.rstride;
      reinterpret_cast<int*>(rb + REC_KEY)[ug & 127] = w0 + 32 * i + lane;
      if (p.hist) atomicAdd(p.hist + ((long long)bb * p.cpb + jb / kSortBlocks) * p.S_k + w0 + 32 * i + lane, 1);
      float* dd = reinterpret_cast<float*>(rb + REC_DIS);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        dd[r * 128 + (ug & 127)] = d[r];
        dmax[r] = fmaxf(dmax[r], fabsf(d[r]));
      }
    }
    base += s_cnt[4];
    __syncthreads();  // the next window rewrites the bitmaps
  }
  const int U = base;
  const int ntiles = max(1, (U + 127) >> 7);
  for (int e = U + tid; e < ntiles * 128; e += UT) {  // padding entries: the zero key row, no weight
    char* rb = p.rec + ((long long)b * p.tcap + (e >> 7)) * p.rstride;
    reinterpret_cast<int*>(rb + REC_KEY)[e & 127] = p.S_k;
    float* dd = reinterpret_cast<float*>(rb + REC_DIS);
#pragma unroll
    for (int r = 0; r < R; ++r) dd[r * 128 + (e & 127)] = 0.f;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) dmax[r] = warp_max(dmax[r]);
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) s_dmax[warp][r] = dmax[r];
  }
  __syncthreads();
  if (tid == 0) {
    float m = 0.f;
    for (int r = 0; r < R; ++r) {
      float d = 0.f;
      for (int x = 0; x < NW; ++x) d = fmaxf(d, s_dmax[x][r]);
      m = fmaxf(m, d * (r < Rb ? s_wmax[r] : 0.f));
    }
    p.binfo[b] = make_int4(ntiles, dz_scale_exponent(m), U, 0);
    __threadfence();
    s_last = atomicAdd(p.done, 1u) == (unsigned)(p.nblocks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  // the last CTA: order the blocks by descending tile count (counting sort)
  __threadfence();
  int* cnt = reinterpret_cast<int*>(us);
  int* cur = cnt + NBUCKET;
  for (int i = tid; i < 2 * NBUCKET; i += UT) cnt[i] = 0;
  __syncthreads();
  for (long long x = tid; x < p.nblocks; x += UT) atomicAdd(&cnt[min(NBUCKET - 1, __ldcg(&p.binfo[x].x))], 1);
  __syncthreads();
  if (warp == 0) {
    constexpr int PER = NBUCKET / 32;
    int sum = 0;
    for (int i = 0; i < PER; ++i) sum += cnt[NBUCKET - 1 - (PER * lane + i)];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int i = 0; i < PER; ++i) {
      const int nt = NBUCKET - 1 - (PER * lane + i);
      cur[nt] = run;
      run += cnt[nt];
    }
  }
  __syncthreads();
  for (long long x = tid; x < p.nblocks; x += UT)
    p.border[atomicAdd(&cur[min(NBUCKET - 1, __ldcg(&p.binfo[x].x))], 1)] = (int)x;
}

// Words of the per-call counter block used by the kernel choice.
constexpr int SEL_FLAG = 2;      // 1: the per-row kernel serves the call, 0: the blocked one
constexpr int SEL_DONE = 3;      // CTA counter of select_kernel
constexpr int SEL_SUMS = 4;      // three 64-bit sums: union tiles, row tiles, rows
constexpr int SCHED_ZERO = kSchedWords;  // words the k conversion kernel zeroes

// Cost model of the two gemm paths, in thousands of cycles per SM, fitted to
// their measured times (uniform top-k 128 ... 2048 over 4096 keys, the causal
// top-1024 rows over 4096 keys, causal top-512 rows on S_q = S_k = 4096): the
// blocked path pays per block of four rows (its union pass, Q copy,
// block-end epilogue) plus per 128-key union tile; the per-row kernel pays
// per row plus per 128-slot tile of the row.  Its dK reductions collide when
// rows share keys (causal prefixes), which the per-tile costs do not see: it
// is chosen only when its estimate is below the blocked one by a margin (the
// causal top-512 rows lose to the blocked kernel at an estimate 13 % lower;
// uniform top-128 rows win at 18 % lower).
constexpr double COST_BLOCK = 30.0, COST_UNION_TILE = 7.82, COST_ROW = 9.08, COST_ROW_TILE = 3.9;
constexpr double ROWS_MARGIN = 1.15;

// Which gemm kernel serves an atomic call without options: on a strided
// sample of blocks, the union's tiles against the rows' own tiles, through
// the cost model above.  One CTA of four warps per sampled block (warp r on
// row r), a bitmap of the keys in shared memory (S_k <= 65536); the last CTA
// writes the choice.  force >= 0 imposes it (a test switch).
__global__ void __launch_bounds__(128) select_kernel(const int32_t* __restrict__ idx, int S_q, int S_k, int L,
                                                     int nbpb, long long stride, unsigned* __restrict__ sched,
                                                     int force) {
  extern __shared__ uint32_t sbm[];  // ceil(S_k / 32) words
  __shared__ unsigned s_cnt[4], s_pop[4];
  // the union pass may start now: it waits for this kernel's completion
  // before it reads the choice
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int words = (S_k + 31) >> 5;
  for (int i = tid; i < words; i += 128) sbm[i] = 0u;
  __syncthreads();
  const long long b = blockIdx.x * stride;
  const int batch = (int)(b / nbpb), t0 = (int)(b % nbpb) * R;
  const int Rb = min(R, S_q - t0);
  unsigned cnt = 0;
  if (warp < Rb) {
    const int32_t* ir = idx + ((long long)batch * S_q + t0 + warp) * L;
    constexpr int NB = 16;  // ids in flight per lane
    for (int j0 = lane; j0 < L; j0 += 32 * NB) {
      int sv[NB];
#pragma unroll
      for (int k = 0; k < NB; ++k) sv[k] = j0 + 32 * k < L ? __ldg(ir + j0 + 32 * k) : -1;
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        if ((unsigned)sv[k] < (unsigned)S_k) {
          atomicOr(&sbm[sv[k] >> 5], 1u << (sv[k] & 31));
          ++cnt;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(FULL, cnt, o);
  __syncthreads();
  unsigned pop = 0;
  for (int i = tid; i < words; i += 128) pop += __popc(sbm[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pop += __shfl_xor_sync(FULL, pop, o);
  if (lane == 0) {
    s_cnt[warp] = cnt;
    s_pop[warp] = pop;
  }
  __syncthreads();
  griddep_wait();  // the counter block is zeroed by the kernel before
  if (tid == 0) {
    const unsigned U = s_pop[0] + s_pop[1] + s_pop[2] + s_pop[3];
    unsigned long long row_tiles = 0;
    for (int r = 0; r < Rb; ++r) row_tiles += max(1u, (s_cnt[r] + 127u) / 128u);
    unsigned long long* sums = reinterpret_cast<unsigned long long*>(sched + SEL_SUMS);
    atomicAdd(sums, (unsigned long long)max(1u, (U + 127u) / 128u));
    atomicAdd(sums + 1, row_tiles);
    atomicAdd(sums + 2, (unsigned long long)Rb);
    __threadfence();
    if (atomicAdd(sched + SEL_DONE, 1u) == gridDim.x - 1) {
      __threadfence();
      const double ut = (double)__ldcg(sums), rt = (double)__ldcg(sums + 1), nr = (double)__ldcg(sums + 2);
      const double t_blocked = gridDim.x * COST_BLOCK + ut * COST_UNION_TILE;
      const double t_rows = nr * COST_ROW + rt * COST_ROW_TILE;
      sched[SEL_FLAG] = force >= 0 ? (unsigned)force : (ROWS_MARGIN * t_rows < t_blocked ? 1u : 0u);
    }
  }
}

// Dense blocks: block b holds keys [0, t0 + Rb); its dz scale exponent from
// max |dI| over each row's causal keys and max |w|, written to binfo (the
// gemm kernel's scan reads it).  One CTA of four warps per block, warp r on
// row r.
__global__ void __launch_bounds__(128) dense_scale_kernel(const float* __restrict__ dI, const float* __restrict__ w,
                                                          int4* __restrict__ binfo, int S, int H, int nbpb) {
  __shared__ float s_m[4];
  griddep_launch_dependents();
  griddep_wait();  // dI is the score-grad's output
  const long long b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int batch = (int)(b / nbpb), t0 = (int)(b % nbpb) * R;
  const int Rb = min(R, S - t0);
  float m = 0.f;
  if (warp < Rb) {
    const long long row = (long long)batch * S + t0 + warp;
    const float* dr = dI + row * S;
    const int n = t0 + warp + 1;  // causal keys 0 .. t
    float mx = 0.f;
    if ((S & 3) == 0) {
      const float4* d4 = reinterpret_cast<const float4*>(dr);
      for (int v = lane; v < (n >> 2); v += 32) {
        const float4 x = __ldg(d4 + v);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
      }
      for (int j = ((n >> 2) << 2) + lane; j < n; j += 32) mx = fmaxf(mx, fabsf(__ldg(dr + j)));
    } else {
      for (int j = lane; j < n; j += 32) mx = fmaxf(mx, fabsf(__ldg(dr + j)));
    }
    float wm = 0.f;
    for (int h = lane; h < H; h += 32) wm = fmaxf(wm, fabsf(__ldg(w + row * H + h)));
    m = warp_max(mx) * warp_max(wm);
  }
  if (lane == 0) s_m[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    const float mb = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
    const int U = t0 + Rb;
    binfo[b] = make_int4((U + kBM - 1) / kBM, dz_scale_exponent(mb), U, 0);
  }
}

// k (bf16, [B, S_k, D]) -> fp16 [B][S_k + 1][128]: zero padded beyond D, and
// row S_k of each batch zero (padding entries of a tile copy it).
// Launched programmatically after the score-grad kernel (which writes neither
// k nor the workspace), it runs alongside it and waits for it before exiting,
// so that its own completion implies the score-grad's.
__global__ void k_to_f16_kernel(const uint16_t* __restrict__ k, __half* __restrict__ k16, int B, int S_k, int D,
                                unsigned* __restrict__ sched, int nsched, unsigned* __restrict__ status,
                                int* __restrict__ zero32, long long nzero32) {
  griddep_launch_dependents();  // the next kernel may start its prologue
  if (blockIdx.x == 0 && threadIdx.x < nsched) sched[threadIdx.x] = 0u;  // the following kernels' counters
  const long long rows = (long long)B * (S_k + 1);
  const long long n = rows * (kDP / 8);
  bool bad = false;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < n;
       x += (long long)gridDim.x * blockDim.x) {
    const int ch = (int)(x % (kDP / 8));
    const long long row = x / (kDP / 8);
    const int b = (int)(row / (S_k + 1));
    const int s = (int)(row % (S_k + 1));
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (s < S_k && ch * 8 < D) val = __ldg(reinterpret_cast<const uint4*>(k + ((long long)b * S_k + s) * D + ch * 8));
    bad |= bf16x2_out_of_fp16(val.x) || bf16x2_out_of_fp16(val.y) || bf16x2_out_of_fp16(val.z) ||
           bf16x2_out_of_fp16(val.w);
    *reinterpret_cast<uint4*>(k16 + row * kDP + ch * 8) =
        make_uint4(bf16x2_to_half2(val.x), bf16x2_to_half2(val.y), bf16x2_to_half2(val.z), bf16x2_to_half2(val.w));
  }
  // the deterministic sort's per-chunk key counts start at zero
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < nzero32;
       x += (long long)gridDim.x * blockDim.x)
    zero32[x] = 0;
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, DEV_FP16_RANGE);
  griddep_wait();
}

// The final fp32 dK -> bf16 (round to nearest even), 8 values per thread step.
__global__ void dk_to_bf16_kernel(const float* __restrict__ dk, uint16_t* __restrict__ out, long long n) {
  const long long n8 = n / 8;  // n = B*S_k*D, D a multiple of 8
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < n8; x += (long long)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(dk)[2 * x];
    const float4 b = reinterpret_cast<const float4*>(dk)[2 * x + 1];
    uint4 o;
    o.x = (uint32_t)to_bf16(a.x) | ((uint32_t)to_bf16(a.y) << 16);
    o.y = (uint32_t)to_bf16(a.z) | ((uint32_t)to_bf16(a.w) << 16);
    o.z = (uint32_t)to_bf16(b.x) | ((uint32_t)to_bf16(b.y) << 16);
    o.w = (uint32_t)to_bf16(b.z) | ((uint32_t)to_bf16(b.w) << 16);
    reinterpret_cast<uint4*>(out)[x] = o;
  }
}

// Key window of the union pass and the dedup capacity per row (both bounded
// so that its shared memory stays under ~104 KB for any shape), and whether
// the block's id rows (rows of up to 2048 slots) and dI rows (up to 1024) are
// staged in shared memory.
void union_geometry(int S_k, int L, int& W, int& dcap, int& staged, int& staged_dI) {
  const long long skr = ((long long)S_k + 1023) / 1024 * 1024;
  W = (int)std::min<long long>(skr, L <= 4096 ? 32768 : 4096);
  dcap = std::min(L, W);
  staged = L <= 2048 ? 1 : 0;
  staged_dI = L <= 1024 ? 1 : 0;
}

size_t union_smem_bytes(int W, int dcap, int L, int staged, int staged_dI) {
  size_t s = (size_t)10 * (W / 32) * 4 + (size_t)R * dcap * 4;
  if (staged) s += (size_t)(staged_dI ? 2 : 1) * R * ((L + 3) & ~3) * 4;
  return std::max<size_t>(s, 2 * NBUCKET * 4);
}

// Test of the timeout path: IBWD_TEST_TIMEOUT_NS=<ns> in the environment makes
// the record producer of every CTA publish nothing, so that every other role
// waits on a barrier phase that never completes, and shortens the roles' wait
// limit to <ns> (1000 to 2e9).  The waits then run out without any fault; the
// drains of copies and MMAs already issued keep the full 2 s limit.  Returns
// 0 when unset.
unsigned long long test_timeout_ns() {
  const char* v = std::getenv("IBWD_TEST_TIMEOUT_NS");
  if (!v || !*v) return 0;
  const unsigned long long ns = std::strtoull(v, nullptr, 10);
  return ns < 1000 ? 1000 : (ns > 2000000000ull ? 2000000000ull : ns);
}
std::atomic<int> g_attr_union[64];

// q as the gemm kernel's TMA source: a 4-d bf16 tensor [B][S_q][H][D] (D
// innermost), boxes of 4 rows x 64 heads x 64 columns, the 128-byte swizzle;
// elements past S_q, H or D read as zero.  The encoder is the driver's,
// reached through the runtime (no link against the driver library).
bool encode_q_map(CUtensorMap* m, const uint16_t* q, int B, int S_q, int H, int D) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::atomic<int> state{0};  // 0 not looked up, 1 found, 2 missing
  int st = state.load(std::memory_order_acquire);
  if (st == 0) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult res{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &res) ==
            cudaSuccess &&
        res == cudaDriverEntryPointSuccess && fn) {
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      st = 1;
    } else {
      st = 2;
    }
    state.store(st, std::memory_order_release);
  }
  if (st != 1) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S_q, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)S_q * H * D * 2};
  const cuuint32_t box[4] = {64, 64, (cuuint32_t)R, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(q), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Test of the pipeline's ordering: IBWD_TEST_SHALLOW_PIPELINE=1 in the
// environment runs the gemm kernel built with one K-tile stage and two
// tile-record slots instead of two and four; its results must be bitwise
// those of the production depths.
bool test_shallow_pipeline() {
  const char* v = std::getenv("IBWD_TEST_SHALLOW_PIPELINE");
  return v && v[0] == '1';
}

// Test of both gemm kernels on calls the choice covers:
// IBWD_TEST_GEMM_PATH=rows imposes the per-row kernel, =blocked the blocked
// one (no choice is made).  -1: the cost model decides; 0: blocked; 1: rows.
int test_gemm_path() {
  const char* v = std::getenv("IBWD_TEST_GEMM_PATH");
  if (!v) return -1;
  if (std::strcmp(v, "rows") == 0) return 1;
  if (std::strcmp(v, "blocked") == 0) return 0;
  return -1;
}

}  // namespace

cudaError_t launch_k_to_f16(const uint16_t* k, __half* k16, int B, int S_k, int D, unsigned* sched, int nsched,
                            unsigned* status, bool pdl, int num_sms, cudaStream_t st, int* zero32, long long nzero32) {
  const long long n = std::max<long long>((long long)B * (S_k + 1) * (kDP / 8), nzero32);
  const int blocks = (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, 8LL * num_sms));
  return launch_ex(k_to_f16_kernel, (unsigned)blocks, 256u, 0, st, pdl, k, k16, B, S_k, D, sched, nsched, status,
                   zero32, nzero32);
}

WsLayout gemm_workspace_layout(int B, int S_q, int S_k, int H, int D, int L, int deterministic, int dense) {
  (void)H;
  WsLayout w{};
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  w.nbpb = (S_q + R - 1) / R;
  w.nblocks = (long long)B * w.nbpb;
  size_t off = 0;
  w.sched = off;
  off = up(off + 256);
  w.k16 = off;
  off = up(off + (size_t)B * (S_k + 1) * kDP * 2);
  w.binfo = off;
  off = up(off + (size_t)w.nblocks * 16);
  if (!dense) {
    const long long ucap = std::min<long long>(S_k, (long long)R * L);
    w.tcap = (int)std::max<long long>(1, (ucap + kBM - 1) / kBM);
    w.rstride = deterministic ? (int)REC_BYTES : REC_POS;
    w.border = off;
    off = up(off + (size_t)w.nblocks * 4);
    w.rec = off;
    off = up(off + (size_t)w.nblocks * w.tcap * w.rstride);
  }
  if (deterministic) {
    if (dense) {
      // block j of a batch holds keys [0, 4j + Rb): the entries of a batch
      long long per = 0;
      for (int j = 0; j < w.nbpb; ++j) per += std::min(S_q, R * j + R);
      w.entries_cap = (long long)B * per;
    } else {
      w.entries_cap = w.nblocks * std::min<long long>(S_k, (long long)R * L);
      w.nchunks = (long long)B * ((w.nbpb + kSortBlocks - 1) / kSortBlocks);
    }
    w.u = off;
    off = up(off + (size_t)w.entries_cap * u_row_bytes(D));
    w.hist = off;
    if (!dense) off = up(off + (size_t)w.nchunks * S_k * 4);
    w.key_start = off;
    off = up(off + ((size_t)B * S_k + 1) * 4);
  }
  w.total = off;
  return w;
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  const bool dense = a.idx == nullptr;
  const WsLayout lay = gemm_workspace_layout(a.B, a.S_q, a.S_k, a.H, a.D, a.L, a.deterministic, dense);
  char* ws = static_cast<char*>(a.ws);
  __half* k16 = reinterpret_cast<__half*>(ws + lay.k16);
  unsigned* sched = reinterpret_cast<unsigned*>(ws + lay.sched);
  int4* binfo = reinterpret_cast<int4*>(ws + lay.binfo);
  // The per-row kernel can serve atomic sparse calls without options (and
  // keys that fit select_kernel's bitmap); select_kernel chooses on the
  // device, and every kernel of the path that is not chosen exits at once.
  const int forced = test_gemm_path();
  const bool choose = !a.deterministic && !dense && !a.ids_global && !a.dq16 && !a.dw16 && !a.dk16 &&
                      a.sm_scale == 1.f && a.S_k <= 65536 && forced != 0;
  const unsigned* select = choose ? sched + SEL_FLAG : nullptr;
  // programmatic only right after this library's score-grad kernel: the
  // kernel reads k before it waits for its predecessor
  int* hist = (a.deterministic && !dense) ? reinterpret_cast<int*>(ws + lay.hist) : nullptr;
  // deterministic sparse mode: the key counts start at zero
  const long long nzero = hist ? lay.nchunks * a.S_k : 0LL;
  // the k copy and the choice: on the side stream already forked by a
  // one-call entry point (beside its score-grad), else on the call's stream
  const cudaStream_t pre = a.early_side ? a.side : st;
  cudaError_t e = launch_k_to_f16(a.k, k16, a.B, a.S_k, a.D, sched, SCHED_ZERO, a.status,
                                  a.after_score_grad != 0 && !a.early_side, a.num_sms, pre,
                                  a.deterministic ? reinterpret_cast<int*>(ws + lay.hist) : nullptr, nzero);
  if (e != cudaSuccess) return e;
  if (choose) {
    const long long nsample = std::min<long long>(lay.nblocks, 256);
    const long long stride = lay.nblocks / nsample;
    const size_t sh = (size_t)((a.S_k + 31) / 32) * 4;
    e = launch_ex(select_kernel, (unsigned)nsample, 128u, sh, pre, true, static_cast<const int32_t*>(a.idx), a.S_q,
                  a.S_k, a.L, lay.nbpb, stride, sched, forced);
    if (e != cudaSuccess) return e;
  }
  if (a.early_side) {
    // the union pass reads the choice and the zeroed counters
    e = cudaEventRecord(a.ev_sel, a.side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, a.ev_sel, 0);
    if (e != cudaSuccess) return e;
  }
  if (!dense) {
    UParams u{};
    u.idx = a.idx;
    u.dI = a.dI;
    u.w = a.w;
    u.rec = ws + lay.rec;
    u.binfo = binfo;
    u.border = reinterpret_cast<int*>(ws + lay.border);
    u.done = sched + 1;
    u.nblocks = lay.nblocks;
    u.S_q = a.S_q;
    u.S_k = a.S_k;
    u.H = a.H;
    u.L = a.L;
    u.nbpb = lay.nbpb;
    u.tcap = lay.tcap;
    u.rstride = lay.rstride;
    u.hist = hist;
    u.cpb = (lay.nbpb + kSortBlocks - 1) / kSortBlocks;
    u.ids_global = a.ids_global;
    u.select = select;
    union_geometry(a.S_k, a.L, u.W, u.dcap, u.staged, u.staged_dI);
    const size_t sh = union_smem_bytes(u.W, u.dcap, a.L, u.staged, u.staged_dI);
    // (its static arrays come on top of the dynamic bytes: always raise the limit)
    if (!set_smem_attr((const void*)union_kernel, sh, g_attr_union)) return cudaErrorInvalidValue;
    // it reads the ids before its predecessor completes and dI only after
    e = launch_ex(union_kernel, (unsigned)lay.nblocks, (unsigned)UT, sh, st, true, u);
  } else {
    e = launch_ex(dense_scale_kernel, (unsigned)lay.nblocks, 128u, 0, st, true, static_cast<const float*>(a.dI), a.w,
                  binfo, a.S_q, a.H, lay.nbpb);
  }
  if (e != cudaSuccess) return e;
  if (a.deterministic) {
    e = launch_det_sort(a, lay, st);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap qmap;
  if (!encode_q_map(&qmap, a.q, a.B, a.S_q, a.H, a.D)) return cudaErrorInvalidValue;
  BParams p{};
  p.q = a.q;
  p.k16 = k16;
  p.w = a.w;
  p.dI = a.dI;
  p.rec = dense ? nullptr : ws + lay.rec;
  p.binfo = binfo;
  p.border = dense ? nullptr : reinterpret_cast<const int*>(ws + lay.border);
  p.dq = a.dq;
  p.dw = a.dw;
  p.dk = a.dk;
  p.u = a.deterministic ? ws + lay.u : nullptr;
  p.dq16 = a.dq16;
  p.dw16 = a.dw16;
  p.sched = sched;
  p.status = a.status;
  p.nblocks = lay.nblocks;
  p.drain_ns = 2000000000ull;
  p.sm_scale = a.sm_scale > 0.f ? a.sm_scale : 1.f;
  const unsigned long long test_ns = test_timeout_ns();
  p.wait_ns = test_ns ? test_ns : 2000000000ull;
  p.test_stall = test_ns != 0;
  p.select = select;
  p.B = a.B;
  p.S_q = a.S_q;
  p.S_k = a.S_k;
  p.H = a.H;
  p.D = a.D;
  p.L = a.L;
  p.dense = dense ? 1 : 0;
  p.nbpb = lay.nbpb;
  p.tcap = lay.tcap;
  p.rstride = lay.rstride;
  p.dense_batch_entries = (dense && a.deterministic) ? lay.entries_cap / a.B : 0;
  const int grid = (int)std::min<long long>(a.num_sms, lay.nblocks);
  e = test_shallow_pipeline() ? launch_blk_pipe<1, 2>(p, qmap, grid, st) : launch_blk_pipe<2, 4>(p, qmap, grid, st);
  if (e != cudaSuccess) return e;
  if (choose) {
    // the per-row kernel: runs only if chosen (then the blocked kernel has
    // exited at once); the row counter is the block counter's word
    e = launch_gemm_rows_kernel(a, k16, sched, select, st);
    if (e != cudaSuccess) return e;
  }
  if (a.deterministic) {
    e = launch_det_segsum(a, lay, st);
    if (e != cudaSuccess) return e;
  }
  if (a.dk16) {
    const long long n = (long long)a.B * a.S_k * a.D;
    const int blocks = (int)std::max<long long>(1, std::min<long long>((n / 8 + 255) / 256, 4LL * a.num_sms));
    dk_to_bf16_kernel<<<blocks, 256, 0, st>>>(a.dk, a.dk16, n);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace ibwd
