// Gemm stage of the lightning-indexer backward on sm_103a (kernel 2), with
// the query rows taken in blocks of four.
//
// Definition (cudnn-frontend #730 "optimize SM100 gradient kernels",
// benchmark-harness comment, ref_grads; #549 names the kernel kernel_gemm and
// its outputs d_index_q, d_weights, d_index_k), per query row t and selected
// key s = idx[t,j] (padding ids, i.e. any id outside [0, S_k), are skipped):
//   z[h]    = q[t,h,:] . k[s,:]                       (forward recompute)
//   dW[t,h] = sum_s dI[t,s] relu(z[h])
//   dz[h]   = dI[t,s] w[t,h] [z[h] > 0]
//   dQ[t,h] = sum_s dz[h] k[s,:]
//   dK[s]  += sum_h dz[h] q[t,h,:]
//
// Design.  dK is a scatter of one 512-byte fp32 row per (query row, selected
// key); on this GPU fp32 reductions into L2 top out near 6.5 TB/s whichever
// way they are issued, which makes that scatter the bound of a kernel that
// treats every row on its own.  Adjacent query rows select largely the same
// keys (causal ranges, local windows), so here the unit of work is a BLOCK
// of four consecutive rows of one batch, processed against the UNION of
// their valid keys: the four rows' contributions to a key are summed by the
// tensor core before one reduction per (block, key).  The union is built by
// a pass before the kernel (union_kernel): per block, the keys in ascending
// order, and per (key, row) the sum of that row's dI over its slots
// selecting the key (0 when the row does not select it), in tile records of
// 128 entries.  The tensor-core work per key grows fourfold; the scatter
// shrinks by the union factor (about one half on the causal workloads).
//
// Per 128-entry tile g of a block (keys are its N or M dimension, the four
// rows' 64 heads are 256 "(r,h)" rows):
//   MMA1 (twice) Z[(r,h), s] = Q[(r,h), d] . Ksel[s, d]^T for rows 0-1 and
//                2-3 in turn (M = 128, N = 128, K = 128) into one TMEM buffer
//   MMA3 dQ^T[d, (r,h)] += Ksel^T[d, s] . dz[(r,h), s]^T   (N = 256)
//   MMA2 dK^T[d, s]      = Q^T[d, (r,h)] . dz[(r,h), s]     (K = 256)
// TMEM: Z 128 columns, dK 128, dQ 256 (all 512).  Operands are fp16 in
// 128-byte-swizzled shared memory: k is converted once (bf16 -> fp16 is
// exact in fp16 range), q per block, and dz carries a per-block power-of-two
// scale 2^c that keeps it in the fp16 normal range (a bf16 dz would cost
// ~1.6e-3 relative RMS in dK, over its budget); the scale is undone exactly
// in the fp32 epilogues.  With Z transposed (TMEM lane = (r,h)), a dz thread
// owns one (r,h) for the whole block: dW accumulates in a register over the
// keys, with no cross-lane reduction per tile.
//
// Warp roles (32 warps; a warp reaches TMEM lanes 32*(warp%4) .. +31):
//   0-1   gather: the tile's 128 fp16 key rows by 16-byte cp.async into a
//         K stage (two stages)
//   2     scan: claims blocks, copies each tile record into a shared ring
//         (bulk copy; dense blocks: builds it from dI), publishes the block
//   3     Z MMA issuer (one elected lane) and TMEM owner
//   4     dQ / dK MMA issuer
//   5-7   Q loader: the block's q rows by cp.async, converted to fp16 in
//         place; w
//   8-23  dz: Z -> mask, dW partial, fp16 dz tile; at block end dW and the
//         dQ epilogue (TMEM -> fp32)
//   24-31 dK: dK^T tile from TMEM -> fp32 red.global.add (one 128-byte line
//         per warp-instruction lane group) into dk, or plain stores of the
//         entry's row into u at its sorted position (deterministic mode)
// Every mbarrier wait is bounded: on expiry the kernel raises a status bit,
// all roles unwind, in-flight copies and MMAs are drained and TMEM is freed.
#include <algorithm>
#include <atomic>
#include <climits>

#include "kcommon.cuh"

namespace ibwd {
namespace {

constexpr int R = kBlkRows;   // query rows per block
constexpr int NR = R * kHP;   // (r,h) rows of a block: 256
constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------ union pass --
constexpr int UT = 128;        // threads: warp r handles row r of the block
constexpr int NBUCKET = 1024;  // tile-count buckets of the block order
constexpr int REC_KEY = 0, REC_DIS = 512, REC_POS = 2560;  // byte offsets in a tile record

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
  int W;       // key window per pass (multiple of 1024)
  int dcap;    // per-row capacity of the dedup arrays: min(L, W)
  int staged;  // the block's ids and dI rows are copied into shared memory (Lp = L rounded up to 4)
};

// Whether a block's dW is summed per key (1) rather than recovered from the
// dQ accumulator: when the smallest |w| of its heads is zero, below 2^-12 of
// the largest, or not finite.
__device__ __forceinline__ int direct_dw(float wmin, float wmax) {
  return (wmin > 0.f && wmin >= 0x1p-12f * wmax && wmax <= 3.0e38f) ? 0 : 1;
}

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
// values in lane order, steps in slot order, so the sum is fixed); then the
// union's entries are written in ascending key order with the four rows'
// sums.  The largest |dis| * |w| of the block fixes its dz scale.  The last
// CTA to finish orders all blocks by descending tile count (a processing
// order for the gemm kernel; it affects no result).
__global__ void __launch_bounds__(UT) union_kernel(const UParams p) {
  extern __shared__ __align__(16) uint32_t us[];
  const int WW = p.W >> 5;
  const int Lp = (p.L + 3) & ~3;
  uint32_t* bm = us;                                      // [5][WW]: rows 0-3, union
  int* pf = reinterpret_cast<int*>(us + 5 * WW);          // [5][WW]
  float* drow = reinterpret_cast<float*>(us + 10 * WW);   // [4][dcap]
  int* ids_s = reinterpret_cast<int*>(drow + R * p.dcap);  // staged: [4][Lp] ids, then [4][Lp] dI
  float* dI_s = reinterpret_cast<float*>(ids_s + R * Lp);
  __shared__ int s_cnt[5], s_kmin[4], s_kmax[4];
  __shared__ float s_wmax[4], s_wmin[4], s_dmax[4][R];
  __shared__ int s_last;
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long b = blockIdx.x;
  const int bb = (int)(b / p.nbpb), jb = (int)(b % p.nbpb);
  const int t0 = jb * R;
  const int Rb = min(R, p.S_q - t0);
  const long long row0 = (long long)bb * p.S_q + t0;
  const unsigned off = p.ids_global ? (unsigned)bb * (unsigned)p.S_k : 0u;  // rows < 2^31
  const bool own = warp < Rb;
  // this warp's row: in shared memory when staged, else global
  const int32_t* ir = p.staged ? ids_s + warp * Lp : p.idx + (own ? (row0 + warp) * p.L : 0);
  const float* dr_in = p.staged ? dI_s + warp * Lp : p.dI + (own ? (row0 + warp) * p.L : 0);
  if (p.staged) stage_rows(smem_u32(ids_s), p.idx, row0, Rb, p.L, Lp);

  float wmax = 0.f, wmin = 3.0e38f;  // over the row's heads; wmin stays large for rows past the block
  if (own) {
    for (int h = lane; h < p.H; h += 32) {
      const float a = fabsf(__ldg(p.w + (row0 + warp) * p.H + h));
      wmax = fmaxf(wmax, a);
      wmin = fminf(wmin, a);
    }
    wmax = warp_max(wmax);
    wmin = -warp_max(-wmin);
  }
  if (p.staged) {
    cp_async_wait_all();
    __syncthreads();
  }
  // key range of the block's valid slots (one window covers every key when S_k <= W)
  int kmin = 0, kmax = p.S_k - 1;
  if (p.S_k > p.W) {
    kmin = INT_MAX;
    kmax = -1;
    if (own) {
      for (int j = lane; j < p.L; j += 32) {
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
  if (lane == 0) {
    s_wmax[warp] = wmax;
    s_wmin[warp] = wmin;
  }
  __syncthreads();
  if (p.S_k > p.W) {
    kmin = min(min(s_kmin[0], s_kmin[1]), min(s_kmin[2], s_kmin[3]));
    kmax = max(max(s_kmax[0], s_kmax[1]), max(s_kmax[2], s_kmax[3]));
  }
  // dI is written by the kernel before this one (score-grad)
  griddep_wait();
  if (p.staged) {
    stage_rows(smem_u32(dI_s), p.dI, row0, Rb, p.L, Lp);
    cp_async_wait_all();
    __syncthreads();
  }

  float dmax[R] = {0.f, 0.f, 0.f, 0.f};
  int base = 0;
  for (long long w0l = kmin; w0l <= kmax; w0l += p.W) {  // no pass when the block has no valid slot
    const int w0 = (int)w0l;
    for (int i = tid; i < 5 * WW; i += UT) bm[i] = 0u;
    __syncthreads();
    bool dup = false;
    if (own) {
      for (int j = lane; j < p.L; j += 32) {
        const int s = (int)((unsigned)ir[j] - off);
        const unsigned x = (unsigned)(s - w0);
        if ((unsigned)s < (unsigned)p.S_k && x < (unsigned)p.W) {
          const uint32_t bit = 1u << (x & 31);
          const uint32_t old = atomicOr(&bm[warp * WW + (x >> 5)], bit);
          dup |= (old & bit) != 0u;
        }
      }
    }
    dup = __any_sync(FULL, dup);
    __syncthreads();
    for (int i = tid; i < WW; i += UT) bm[4 * WW + i] = bm[i] | bm[WW + i] | bm[2 * WW + i] | bm[3 * WW + i];
    __syncthreads();
    for (int x = warp; x < 5; x += UT / 32) {
      const int n = warp_popc_prefix(bm + x * WW, pf + x * WW, WW);
      if (lane == 0) s_cnt[x] = n;
    }
    __syncthreads();
    if (own) {
      float* drr = drow + warp * p.dcap;
      const uint32_t* bmr = bm + warp * WW;
      const int* pfr = pf + warp * WW;
      if (dup) {
        for (int i = lane; i < s_cnt[warp]; i += 32) drr[i] = 0.f;
        __syncwarp();
      }
      for (int j0 = 0; j0 < p.L; j0 += 32) {
        const int j = j0 + lane;
        int rank = -1;
        float v = 0.f;
        if (j < p.L) {
          const int s = (int)((unsigned)ir[j] - off);
          const unsigned x = (unsigned)(s - w0);
          if ((unsigned)s < (unsigned)p.S_k && x < (unsigned)p.W) {
            rank = pfr[x >> 5] + __popc(bmr[x >> 5] & ((1u << (x & 31)) - 1u));
            v = dr_in[j];
          }
        }
        if (!dup) {
          if (rank >= 0) drr[rank] = v;
        } else {
          const unsigned grp = __match_any_sync(FULL, rank >= 0 ? rank : -1 - lane);
          float sum = 0.f;
          for (int l = 0; l < 32; ++l) {
            const float y = __shfl_sync(FULL, v, l);
            if ((grp >> l) & 1u) sum += y;
          }
          if (rank >= 0 && (grp & ((1u << lane) - 1u)) == 0u) drr[rank] += sum;
          __syncwarp();
        }
      }
    }
    __syncthreads();
    // the union's entries of this window, in ascending key order: a warp
    // takes one bitmap word at a time and lane l its bit l, so the set lanes
    // write consecutive entries
    for (int i = warp; i < WW; i += UT / 32) {
      const uint32_t m = bm[4 * WW + i];
      if (!((m >> lane) & 1u)) continue;
      const uint32_t below = (1u << lane) - 1u;
      const int ug = base + pf[4 * WW + i] + __popc(m & below);
      char* rb = p.rec + ((long long)b * p.tcap + (ug >> 7)) * p.rstride;
      reinterpret_cast<int*>(rb + REC_KEY)[ug & 127] = w0 + 32 * i + lane;
      float* dd = reinterpret_cast<float*>(rb + REC_DIS);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t mr = bm[r * WW + i];
        const float d = ((mr >> lane) & 1u) ? drow[r * p.dcap + pf[r * WW + i] + __popc(mr & below)] : 0.f;
        dd[r * 128 + (ug & 127)] = d;
        dmax[r] = fmaxf(dmax[r], fabsf(d));
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
    float m = 0.f, wx = 0.f, wn = 3.0e38f;
    for (int r = 0; r < R; ++r) {
      const float d = fmaxf(fmaxf(s_dmax[0][r], s_dmax[1][r]), fmaxf(s_dmax[2][r], s_dmax[3][r]));
      m = fmaxf(m, d * s_wmax[r]);
      wx = fmaxf(wx, s_wmax[r]);
      wn = fminf(wn, s_wmin[r]);
    }
    p.binfo[b] = make_int4(ntiles, dz_scale_exponent(m), U, direct_dw(wn, wx));
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

// ----------------------------------------------------------- gemm kernel --
constexpr int KST = 2;  // K-tile stages
constexpr int MST = 4;  // tile-record ring
constexpr int BQ = 4;   // block ring (scan -> Q loader)
constexpr int NTHREADS = 1024;
constexpr int W_GATHER0 = 0, W_SCAN = 2, W_MMA = 3, W_GMMA = 4, W_Q0 = 5, W_DZ0 = 8, W_DK0 = 24;
constexpr int NGT = 64, NQT = 96, NDZT = 512, NDKT = 256;
constexpr int NKQ = 4;  // key quarters of a tile: four dz warps per TMEM lane quarter

constexpr uint32_t KTILE = kBM * kDP * 2;  // 32 KB: [2 d-halves][128 keys][128 B]
constexpr uint32_t KHALF = kBM * 128;      // 16 KB
constexpr uint32_t QDH = NR * 128;         // Q block, one 64-d half: [256 (r,h)][128 B] = 32 KB
constexpr uint32_t DZKC = NR * 128;        // dz tile, one 64-key chunk: [256 (r,h)][128 B] = 32 KB
constexpr uint32_t REC_BYTES = 3072;       // one tile record in shared memory

constexpr uint32_t TM_Z = 0, TM_DK = 128, TM_DQ = 256, TM_COLS = 512;

enum { F_FIRST = 1, F_LAST = 2, F_END = 4 };

struct Hdr {        // per tile, written by the scan
  int row0;         // global row index of the block's first row
  int Rb;           // rows in the block (1..4)
  int count;        // entries in the tile (the rest are padding)
  int c;            // dz scale exponent of the block
  int flags;
  int batch;
  int direct;       // dW of this block by per-key accumulation (some |w| is zero or tiny)
  int pad;
};

struct Bars {
  uint64_t kfull[KST], kempty[KST];
  uint64_t mfull[MST], mempty[MST];
  uint64_t bfull[BQ], bempty[BQ];
  uint64_t qfull, qempty;
  uint64_t zfull, zempty;
  uint64_t dzfull, dzempty;
  uint64_t dkfull, dkempty;
  uint64_t dqfull, dqempty;
  uint64_t dwbar;
  uint64_t drain;
};

constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = OFF_K + KST * KTILE;
constexpr uint32_t OFF_DZ = OFF_Q + 2 * QDH;
constexpr uint32_t OFF_REC = OFF_DZ + 2 * DZKC;
constexpr uint32_t OFF_HDR = OFF_REC + MST * REC_BYTES;
constexpr uint32_t OFF_W = OFF_HDR + MST * sizeof(Hdr);      // [4 rows][64 heads] fp32
constexpr uint32_t OFF_DWP = OFF_W + NR * 4;                 // dW partials [4][256]
constexpr uint32_t OFF_DKST = OFF_DWP + NKQ * NR * 4;        // dK transpose stages, 2 KB per dK warp
constexpr uint32_t OFF_BQ = OFF_DKST + (NDKT / 32) * 2048;   // int4 per block ring slot
constexpr uint32_t OFF_BARS = OFF_BQ + BQ * 16;
constexpr uint32_t OFF_MISC = OFF_BARS + sizeof(Bars);
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;        // + alignment slack
static_assert(OFF_BARS % 8 == 0 && OFF_REC % 1024 == 0 && OFF_DZ % 1024 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct BParams {
  const uint16_t* q;   // bf16 [rows, H, D]
  const __half* k16;   // [B][S_k + 1][128]; row S_k of each batch is zero
  const float* w;      // [rows, H]
  const float* dI;     // dense: [rows, S] (sparse blocks read their tile records instead)
  const char* rec;     // sparse: tile records
  const int4* binfo;   // sparse: per block {tiles, c, entries, 0}
  const int* border;   // sparse: processing order of the blocks
  float* dq;
  float* dw;
  float* dk;           // [B, S_k, D] (atomic mode)
  float* u;            // deterministic: per-entry dK rows in key order, or nullptr
  uint16_t* dq16;      // bf16 outputs instead of dq / dw when set
  uint16_t* dw16;
  unsigned* sched;     // block counter, zeroed by the k conversion kernel
  unsigned* status;
  long long nblocks;
  unsigned long long wait_ns;
  int B, S_q, S_k, H, D, L;
  int dense, nbpb, tcap, rstride;
  long long dense_batch_entries;  // deterministic dense: entries (rows of u) per batch
};

struct Ctx {
  uint32_t sbase;
  uint8_t* smem;
  Bars* bars;
  Hdr* hdr;
  volatile int* abort;
  uint32_t tmem;
};

__device__ __forceinline__ const int* rec_key(const Ctx& cx, int ms) {
  return reinterpret_cast<const int*>(cx.smem + OFF_REC + ms * REC_BYTES + REC_KEY);
}
__device__ __forceinline__ const float* rec_dis(const Ctx& cx, int ms) {
  return reinterpret_cast<const float*>(cx.smem + OFF_REC + ms * REC_BYTES + REC_DIS);
}
__device__ __forceinline__ const int* rec_pos(const Ctx& cx, int ms) {
  return reinterpret_cast<const int*>(cx.smem + OFF_REC + ms * REC_BYTES + REC_POS);
}

#define WAIT(bar, par) mbar_wait((bar), (uint32_t)(par), cx.abort, p.status, p.wait_ns)
// Warp-uniform form for the MMA warp, which must stay converged (elect.sync).
#define WAITW(bar, par) __all_sync(FULL, WAIT(bar, par))

// Optional per-tile timeline (clock64 stamps of each role's progress in the
// first CTAs), compiled only with -DIBWD_TRACE for pipeline analysis.
enum TraceEv {
  EV_SCAN_PUB, EV_GATHER_ISSUED, EV_MMA_ZA, EV_MMA_ZB, EV_MMA_DQ, EV_MMA_DK, EV_DZ_ZA, EV_DZ_ZB, EV_DZ_DONE,
  EV_DK_FULL, EV_DK_DONE, EV_Q_START, EV_Q_DONE, EV_COUNT
};
#ifdef IBWD_TRACE
constexpr int TRACE_CTAS = 4, TRACE_TILES = 512;
__device__ unsigned long long g_trace[TRACE_CTAS][EV_COUNT][TRACE_TILES];
constexpr int TRACE_ALL = 1024;
__device__ unsigned long long g_trace_cta[TRACE_ALL][4];  // clock64 start, end; tiles; blocks
#define TRACE(ev, g)                                                                                      \
  do {                                                                                                    \
    if (blockIdx.x < TRACE_CTAS && (g) >= 0 && (g) < TRACE_TILES) g_trace[blockIdx.x][ev][g] = clock64(); \
  } while (0)
#define TRACE_CTA(i, v)                                                   \
  do {                                                                    \
    if (blockIdx.x < TRACE_ALL) g_trace_cta[blockIdx.x][i] = (v);         \
  } while (0)
#else
#define TRACE(ev, g) \
  do {               \
  } while (0)
#define TRACE_CTA(i, v) \
  do {                  \
  } while (0)
#endif

// Dense blocks in descending work: the last blocks of each batch first.
__device__ __forceinline__ long long dense_block_at(const BParams& p, long long pos) {
  const long long jb = p.nbpb - 1 - pos / p.B;
  return (pos % p.B) * p.nbpb + jb;
}

// Deterministic dense mode: the row of u of key s in block jb of a batch.
// Key s lies in blocks floor(s/4) .. nbpb-1; before it come the keys s' < s,
// nbpb - floor(s'/4) entries each.
__device__ __forceinline__ long long dense_pos(const BParams& p, int batch, int s, int jb) {
  const long long a = s >> 2, c = s & 3;
  const long long before = (long long)s * p.nbpb - (2 * a * (a - 1) + c * a);
  return (long long)batch * p.dense_batch_entries + before + (jb - a);
}

// ----------------------------------------------------------------- scan ---
__device__ void scan_role(const BParams& p, const Ctx& cx) {
  const int lane = threadIdx.x & 31;
  Bars* B = cx.bars;
  int4* bq = reinterpret_cast<int4*>(cx.smem + OFF_BQ);
  const uint32_t copy_bytes = p.u ? REC_BYTES : (uint32_t)REC_POS;
  long long g = 0, i = 0;
  long long pos = blockIdx.x;  // the grid never exceeds the block count
  for (;; ++i) {
    const long long b = p.dense ? dense_block_at(p, pos) : (long long)__ldg(p.border + pos);
    const int batch = (int)(b / p.nbpb), jb = (int)(b % p.nbpb);
    const int t0 = jb * R;
    const int Rb = min(R, p.S_q - t0);
    const int row0 = batch * p.S_q + t0;
    int ntiles, c, U, direct;
    if (!p.dense) {
      const int4 bi = __ldg(p.binfo + b);
      ntiles = bi.x;
      c = bi.y;
      U = bi.z;
      direct = bi.w;
    } else {
      // keys [0, t0 + Rb); the scale from max |dI| over each row's causal keys and max |w|
      U = t0 + Rb;
      ntiles = (U + kBM - 1) / kBM;
      float m = 0.f, wx = 0.f, wn = 3.0e38f;
      for (int r = 0; r < Rb; ++r) {
        const float* dr = p.dI + (long long)(row0 + r) * p.S_q;
        const int n = t0 + r + 1;
        float mx = 0.f;
        if ((p.S_q & 3) == 0) {
          const float4* d4 = reinterpret_cast<const float4*>(dr);
          const int n4 = n >> 2;
          int v = lane;
          for (; v + 96 < n4; v += 128) {
            float4 x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = __ldg(d4 + v + 32 * k);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x[k].x), fabsf(x[k].y)), fmaxf(fabsf(x[k].z), fabsf(x[k].w))));
          }
          for (; v < n4; v += 32) {
            const float4 x = __ldg(d4 + v);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
          }
          for (int j = 4 * n4 + lane; j < n; j += 32) mx = fmaxf(mx, fabsf(__ldg(dr + j)));
        } else {
          for (int j = lane; j < n; j += 32) mx = fmaxf(mx, fabsf(__ldg(dr + j)));
        }
        float wm = 0.f, wl = 3.0e38f;
        for (int h = lane; h < p.H; h += 32) {
          const float a = fabsf(__ldg(p.w + (long long)(row0 + r) * p.H + h));
          wm = fmaxf(wm, a);
          wl = fminf(wl, a);
        }
        wm = warp_max(wm);
        m = fmaxf(m, warp_max(mx) * wm);
        wx = fmaxf(wx, wm);
        wn = fminf(wn, -warp_max(-wl));
      }
      c = dz_scale_exponent(m);
      direct = direct_dw(wn, wx);
    }
    // publish the block to the Q loader; warm L2 with its q rows
    if (!WAIT(&B->bempty[i % BQ], ((i / BQ) & 1) ^ 1)) return;
    if (lane == 0) {
      bq[i % BQ] = make_int4(row0, Rb, 0, 0);
      mbar_arrive(&B->bfull[i % BQ]);
      const uint32_t qbytes = (uint32_t)Rb * p.H * p.D * 2;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.q + (long long)row0 * p.H * p.D),
                   "r"(qbytes)
                   : "memory");
    }
    unsigned pend = 0;
    bool last_blk = false;
    long long next = 0;
    for (int k = 0; k < ntiles; ++k, ++g) {
      if (k == 0 && lane == 0) pend = atomicAdd(p.sched, 1u);  // claim the next block now, resolve at the end
      if (k == ntiles - 1) {
        next = (long long)gridDim.x + __shfl_sync(FULL, pend, 0);
        last_blk = next >= p.nblocks;
      }
      const int ms = (int)(g % MST);
      if (!WAIT(&B->mempty[ms], ((g / MST) & 1) ^ 1)) return;
      const int count = min(kBM, U - k * kBM);
      const int flags = (k == 0 ? F_FIRST : 0) | (k == ntiles - 1 ? F_LAST : 0) | (last_blk ? F_END : 0);
      uint8_t* rs = cx.smem + OFF_REC + ms * REC_BYTES;
      if (!p.dense) {
        if (lane == 0) {
          cx.hdr[ms] = Hdr{row0, Rb, max(count, 0), c, flags, batch, direct, 0};
          fence_proxy_async_smem();  // earlier generic reads of the slot precede the async writes
          mbar_arrive_expect_tx(&B->mfull[ms], copy_bytes);
          bulk_g2s(smem_u32(rs), p.rec + ((long long)b * p.tcap + k) * p.rstride, copy_bytes, &B->mfull[ms]);
          TRACE(EV_SCAN_PUB, g);
        }
      } else {
        int* key = reinterpret_cast<int*>(rs + REC_KEY);
        float* dis = reinterpret_cast<float*>(rs + REC_DIS);
        int* pos_s = reinterpret_cast<int*>(rs + REC_POS);
        float v[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int m4 = 0; m4 < 4; ++m4) {
            const int s = k * kBM + lane + 32 * m4;
            v[r][m4] = (r < Rb && s <= t0 + r) ? __ldg(p.dI + (long long)(row0 + r) * p.S_q + s) : 0.f;
          }
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const int e = lane + 32 * m4, s = k * kBM + e;
          key[e] = s < U ? s : p.S_k;
#pragma unroll
          for (int r = 0; r < R; ++r) dis[r * kBM + e] = v[r][m4];
          if (p.u) pos_s[e] = s < U ? (int)dense_pos(p, batch, s, jb) : 0;
        }
        __syncwarp();
        if (lane == 0) {
          cx.hdr[ms] = Hdr{row0, Rb, count, c, flags, batch, direct, 0};
          mbar_arrive(&B->mfull[ms]);
        }
      }
    }
    if (last_blk) break;
    pos = next;
  }
  // end of the block list for the Q loader
  ++i;
  if (!WAIT(&B->bempty[i % BQ], ((i / BQ) & 1) ^ 1)) return;
  if (lane == 0) {
    bq[i % BQ] = make_int4(-1, 0, 0, 0);
    mbar_arrive(&B->bfull[i % BQ]);
  }
}

// --------------------------------------------------------------- gather ---
// Thread x copies chunk (x % 16) of entries (x / 16) + 4i, i = 0..31: every
// warp instruction moves two whole 256-byte key rows.  Row e of the tile
// lands in the 128-byte-swizzle layout: half (chunk / 8), XOR (chunk % 8) ^
// (e % 8).  Each thread's copies arrive on the stage barrier when they land.
__device__ void gather_role(const BParams& p, const Ctx& cx) {
  const int x = threadIdx.x - W_GATHER0 * 32;  // 0..63
  const int rsub = x >> 4, ch = x & 15;
  // rows rsub + 4i: (row % 8) alternates between rsub and rsub + 4
  const uint32_t off0 = (ch >> 3) * KHALF + rsub * 128 + (((ch & 7) ^ rsub) << 4);
  const uint32_t off1 = (ch >> 3) * KHALF + (rsub + 4) * 128 + (((ch & 7) ^ (rsub + 4)) << 4);
  for (int g = 0;; ++g) {
    const int ms = g % MST;
    if (!WAIT(&cx.bars->mfull[ms], (g / MST) & 1)) break;
    const int flags = cx.hdr[ms].flags, batch = cx.hdr[ms].batch;
    const int* keys = rec_key(cx, ms);
    const int st = g % KST;
    if (!WAIT(&cx.bars->kempty[st], ((g / KST) & 1) ^ 1)) break;
    const uint32_t kbase = cx.sbase + OFF_K + st * KTILE;
    const __half* kb = p.k16 + (long long)batch * (p.S_k + 1) * kDP + ch * 8;
#pragma unroll 4
    for (int i2 = 0; i2 < kBM / 8; ++i2) {  // rows rsub + 8*i2 and rsub + 4 + 8*i2
      const int k0 = keys[rsub + 8 * i2], k1 = keys[rsub + 4 + 8 * i2];  // padding entries hold the zero row S_k
      cp_async16(kbase + off0 + i2 * 1024, kb + (long long)k0 * kDP, 16);
      cp_async16(kbase + off1 + i2 * 1024, kb + (long long)k1 * kDP, 16);
    }
    cp_async_mbar_arrive_noinc(&cx.bars->kfull[st]);
    if (x == 0) TRACE(EV_GATHER_ISSUED, g);
    if (flags & F_END) break;
  }
  cp_async_wait_all();  // copies in flight must land before the CTA can exit
}

// ------------------------------------------------------------- Q loader ---
// The block's q rows (bf16) land by cp.async in the fp16 operand's swizzled
// positions ([d-half][(r,h) = 64r + h][128 B]) and are converted in place
// (bf16 -> fp16 keeps the element size); rows past the block, heads past H
// and columns past D are zero.
__device__ void q_role(const BParams& p, const Ctx& cx) {
  const int tid = threadIdx.x - W_Q0 * 32;  // 0..95
  Bars* B = cx.bars;
  const int4* bq = reinterpret_cast<const int4*>(cx.smem + OFF_BQ);
  float* w_s = reinterpret_cast<float*>(cx.smem + OFF_W);
  for (long long i = 0;; ++i) {
    if (!WAIT(&B->bfull[i % BQ], (i / BQ) & 1)) return;
    const int row0 = bq[i % BQ].x, Rb = bq[i % BQ].y;
    mbar_arrive(&B->bempty[i % BQ]);
    if (row0 < 0) return;
    // the previous block's last MMAs that read Q (and its w) are complete
    if (!WAIT(&B->qempty, (i & 1) ^ 1)) return;
    if (tid == 0) TRACE(EV_Q_START, (int)i);
    constexpr int NCHUNK = NR * 16;  // 16-byte chunks of the block
#pragma unroll 4
    for (int x = tid; x < NCHUNK; x += NQT) {
      const int n = x >> 4, c = x & 15, r = n >> 6, h = n & 63;
      const bool ok = r < Rb && h < p.H && c * 8 < p.D;
      const uint16_t* src = ok ? p.q + ((long long)(row0 + r) * p.H + h) * p.D + c * 8 : p.q;
      cp_async16(cx.sbase + OFF_Q + (c >> 3) * QDH + n * 128 + (((c & 7) ^ (n & 7)) << 4), src, ok ? 16u : 0u);
    }
    float wv[(NR + NQT - 1) / NQT];  // w of the block, loaded while the copies fly
#pragma unroll
    for (int k = 0; k < (NR + NQT - 1) / NQT; ++k) {
      const int e = tid + NQT * k, r = e >> 6, h = e & 63;
      wv[k] = (e < NR && r < Rb && h < p.H) ? __ldg(p.w + (long long)(row0 + r) * p.H + h) : 0.f;
    }
    cp_async_wait_all();
#pragma unroll 4
    for (int x = tid; x < NCHUNK; x += NQT) {
      const int n = x >> 4, c = x & 15;
      const uint32_t a = cx.sbase + OFF_Q + (c >> 3) * QDH + n * 128 + (((c & 7) ^ (n & 7)) << 4);
      uint32_t v0, v1, v2, v3;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(a));
      st_shared_v4(a, bf16x2_to_half2(v0), bf16x2_to_half2(v1), bf16x2_to_half2(v2), bf16x2_to_half2(v3));
    }
#pragma unroll
    for (int k = 0; k < (NR + NQT - 1) / NQT; ++k)
      if (tid + NQT * k < NR) w_s[tid + NQT * k] = wv[k];
    fence_proxy_async_smem();
    mbar_arrive(&B->qfull);
    if (tid == 0) TRACE(EV_Q_DONE, (int)i);
  }
}

// ------------------------------------------------------------------ MMA ---
// Z[(r,h), s] = Q[(r,h), d] . Ksel[s, d]^T: A = Q rows (K-major), B = Ksel (K-major)
constexpr uint32_t ID_Z = idesc_f16_f32(128, 128, 0, 0);
// dK^T[d, s] = Q^T[d, (r,h)] . dz[(r,h), s]: A = Q^T (MN-major), B = dz (MN-major: keys contiguous)
constexpr uint32_t ID_DK = idesc_f16_f32(128, 128, 1, 1);
// dQ^T[d, (r,h)] = Ksel^T[d, s] . dz^T[s, (r,h)]: A = Ksel^T (MN-major), B = dz rows (K-major: keys contiguous)
constexpr uint32_t ID_DQ = idesc_f16_f32(128, 256, 1, 0);

// Descriptors are built once per operand; a k-step advances the start address
// field (address >> 4, 14 bits: shared memory stays below 256 KB, so the
// addition never carries out of the field).
__device__ __forceinline__ void mma_z(const Ctx& cx, int st, int half) {
  const uint64_t a0 = sw128_desc(cx.sbase + OFF_Q + half * (QDH / 2), 16, 1024);
  const uint64_t b0 = sw128_desc(cx.sbase + OFF_K + st * KTILE, 16, 1024);
#pragma unroll
  for (int k = 0; k < 8; ++k)  // K = D = 128 in steps of 16
    umma_f16_elect(cx.tmem + TM_Z, a0 + (((k >> 2) * QDH + (k & 3) * 32) >> 4),
                   b0 + (((k >> 2) * KHALF + (k & 3) * 32) >> 4), ID_Z, k > 0);
}

__device__ __forceinline__ void mma_dk(const Ctx& cx) {
  const uint64_t a0 = sw128_desc(cx.sbase + OFF_Q, QDH, 1024);
  const uint64_t b0 = sw128_desc(cx.sbase + OFF_DZ, DZKC, 1024);
#pragma unroll
  for (int k = 0; k < NR / 16; ++k)  // K = 256 (r,h) rows in steps of 16
    umma_f16_elect(cx.tmem + TM_DK, a0 + ((k * 2048) >> 4), b0 + ((k * 2048) >> 4), ID_DK, k > 0);
}

__device__ __forceinline__ void mma_dq(const Ctx& cx, int st, bool first) {
  const uint64_t a0 = sw128_desc(cx.sbase + OFF_K + st * KTILE, KHALF, 1024);
  const uint64_t b0 = sw128_desc(cx.sbase + OFF_DZ, 16, 1024);
#pragma unroll
  for (int k = 0; k < 8; ++k)  // K = 128 keys in steps of 16
    umma_f16_elect(cx.tmem + TM_DQ, a0 + ((k * 2048) >> 4), b0 + (((k >> 2) * DZKC + (k & 3) * 32) >> 4), ID_DQ,
                   (first && k == 0) ? 0u : 1u);
}

// Two issuing warps share the tensor pipe.  The Z issuer runs the Z MMAs of
// every tile (rows 0-1, then rows 2-3, each as soon as the dz warps have
// read the previous Z out of TMEM); the G issuer runs the dQ and dK MMAs of
// a tile once its dz tile is complete (the dK MMA also once the dK warps have
// drained the previous dK), so a slow dK drain holds back only the dK MMA,
// not the recompute of the next tiles.
// A block's next Z waits for its q rows, which the Q loader writes once the
// last dK MMA of the previous block (the last reader of Q) is complete.
__device__ void zmma_role(const BParams& p, const Ctx& cx) {
  Bars* B = cx.bars;
  long long g = 0, i = 0, zi = 0;
  for (;; ++g) {
    const int ms = (int)(g % MST), st = (int)(g % KST);
    if (!WAITW(&B->mfull[ms], (g / MST) & 1)) break;
    const int flags = cx.hdr[ms].flags;
    if ((flags & F_FIRST) && !WAITW(&B->qfull, i & 1)) break;
    if (!WAITW(&B->kfull[st], (g / KST) & 1)) break;
    bool ok = true;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      if (!WAITW(&B->zempty, (zi & 1) ^ 1)) {
        ok = false;
        break;
      }
      // the operands were written by cp.async and generic stores: order them
      // before the tensor core's reads
      fence_proxy_async_smem();
      tc_fence_after();
      mma_z(cx, st, half);
      umma_commit_elect(&B->zfull);
      TRACE(half == 0 ? EV_MMA_ZA : EV_MMA_ZB, (int)g);
      ++zi;
    }
    if (!ok) break;
    if (flags & F_LAST) ++i;
    if (flags & F_END) break;
  }
  // every MMA issued so far completes before TMEM can be released
  __syncwarp();
  umma_commit_elect(&B->drain);
  drain_wait(&B->drain, 0, p.status, p.wait_ns);
  if ((threadIdx.x & 31) == 0) TRACE_CTA(2, (unsigned long long)g + 1);
}

__device__ void gmma_role(const BParams& p, const Ctx& cx) {
  Bars* B = cx.bars;
  long long i = 0;
  for (long long g = 0;; ++g) {
    const int ms = (int)(g % MST), st = (int)(g % KST);
    if (!WAITW(&B->mfull[ms], (g / MST) & 1)) break;
    const int flags = cx.hdr[ms].flags;
    if (!WAITW(&B->dzfull, g & 1)) break;
    if ((flags & F_FIRST) && !WAITW(&B->dqempty, (i & 1) ^ 1)) break;
    tc_fence_after();
    mma_dq(cx, st, (flags & F_FIRST) != 0);
    TRACE(EV_MMA_DQ, (int)g);
    // the key stage: its Z MMAs completed before the dz tile could be written
    umma_commit_elect(&B->kempty[st]);
    if (flags & F_LAST) umma_commit_elect(&B->dqfull);
    if (!WAITW(&B->dkempty, (g & 1) ^ 1)) break;
    tc_fence_after();
    mma_dk(cx);
    TRACE(EV_MMA_DK, (int)g);
    umma_commit_elect(&B->dkfull);
    umma_commit_elect(&B->dzempty);
    if (flags & F_LAST) {
      umma_commit_elect(&B->qempty);
      ++i;
    }
    if (flags & F_END) break;
  }
  __syncwarp();
  umma_commit_elect(&B->drain);
  drain_wait(&B->drain, 0, p.status, p.wait_ns);
}

// ------------------------------------------------------------- dz group ---
// dz warp w (0..15): TMEM lane quarter q = w % 4, key quarter kq = w / 4.  For
// each Z buffer (rows 0-1, then rows 2-3) a thread owns the (r,h) row
// 32q + lane of it and the 32 keys 32kq .. 32kq+31 of every tile: it loads
// their z (16 at a time), releases the buffer after the second load, and
// writes dz = dI w 2^c [z > 0] (fp16) into its 64 bytes of the dz row.
//
// dW.  Summing dz z over the keys gives w 2^c dW, and sum_s dz z =
// q . (sum_s dz k_s) = q . dQraw, the dQ accumulator before its 2^-c scale:
// so dW = (q . dQraw) / (w 2^c), one dot product per (r,h) at block end.
// Blocks where some |w| is zero or below 2^-12 of the block's largest (the
// dz of those heads would lose precision or vanish) accumulate
// dW = sum_s dI relu(z) per key instead (Hdr::direct).
__device__ void dz_epilogue(const BParams& p, const Ctx& cx, int row0, int Rb, int c, int direct, int i,
                            float acc0, float acc1, float wv0, float wv1) {
  const int dzw = (threadIdx.x >> 5) - W_DZ0, q = (threadIdx.x >> 5) & 3, kq = dzw >> 2, lane = threadIdx.x & 31;
  const int tdz = threadIdx.x - W_DZ0 * 32;
  float* dwp = reinterpret_cast<float*>(cx.smem + OFF_DWP);
  if (direct) {  // per-key sums of the four key quarters
    dwp[kq * NR + 32 * q + lane] = acc0;
    dwp[kq * NR + 128 + 32 * q + lane] = acc1;
  }
  if (!WAIT(&cx.bars->dqfull, i & 1)) return;
  tc_fence_after();
  const int d = 32 * q + lane;  // TMEM lane = column of dQ
  const float sc = pow2f(-c);
  const int r = kq;             // dQ columns 64kq .. 64kq+63: the heads of row kq
  const bool rowok = r < Rb;
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    float v[16];
    tmem_ld16(cx.tmem + ((uint32_t)(32 * q) << 16) + TM_DQ + 64 * kq + 16 * cc, v);
    tmem_wait_ld_dep16(v);
    if (cc == 3) {
      tc_fence_before();
      mbar_arrive(&cx.bars->dqempty);
    }
    const int h0 = 16 * cc;
    const long long e0 = ((long long)(row0 + r) * p.H + h0) * p.D + d;
    if (rowok && d < p.D) {
      if (p.dq16) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (h0 + j < p.H) p.dq16[e0 + (long long)j * p.D] = to_bf16(v[j] * sc);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (h0 + j < p.H) p.dq[e0 + (long long)j * p.D] = v[j] * sc;
      }
    }
    if (!direct) {
      // q[r,h,d] dQraw[r,h,d] for this lane's d, then summed over the warp's
      // 32 columns d: four exchange steps and a last add leave head h0 + l
      // summed in lanes l and l + 16
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const bool on = rowok && d < p.D && h0 + j < p.H;
        const float qv = on ? __uint_as_float((uint32_t)__ldg(p.q + e0 + (long long)j * p.D) << 16) : 0.f;
        v[j] *= qv;
      }
#pragma unroll
      for (int step = 0; step < 4; ++step) {
        const int o = 16 >> step, nn = 8 >> step;
        const bool upper = (lane & (o >> 1)) != 0;
#pragma unroll
        for (int k = 0; k < nn; ++k) {
          const float send = upper ? v[k] : v[k + nn];
          const float keep = upper ? v[k + nn] : v[k];
          v[k] = keep + __shfl_xor_sync(FULL, send, o >> 1);
        }
      }
      v[0] += __shfl_xor_sync(FULL, v[0], 16);
      if (lane < 16) dwp[q * NR + r * kHP + h0 + lane] = v[0];
    }
  }
  mbar_arrive(&cx.bars->dwbar);
  if (!WAIT(&cx.bars->dwbar, i & 1)) return;
  if (tdz < NR) {
    const int rr = tdz >> 6, h = tdz & 63;
    if (rr < Rb && h < p.H) {
      // the four partials in a fixed order
      const float s4 = ((dwp[tdz] + dwp[NR + tdz]) + dwp[2 * NR + tdz]) + dwp[3 * NR + tdz];
      // thread tdz holds w of (r,h) = tdz: buffer half tdz / 128
      const float dwv = direct ? s4 : s4 / ((tdz < 128 ? wv0 : wv1) * pow2f(c));
      const long long e = (long long)(row0 + rr) * p.H + h;
      if (p.dw16)
        p.dw16[e] = to_bf16(dwv);
      else
        p.dw[e] = dwv;
    }
  }
}

__device__ void dz_role(const BParams& p, const Ctx& cx) {
  const int dzw = (threadIdx.x >> 5) - W_DZ0, lane = threadIdx.x & 31;
  const int q = (threadIdx.x >> 5) & 3, kq = dzw >> 2;
  const int tdz = threadIdx.x - W_DZ0 * 32;  // 0..511
  const int nrow = 32 * q + lane;            // (r,h) row within a Z buffer
  const float* w_s = reinterpret_cast<const float*>(cx.smem + OFF_W);
  Bars* B = cx.bars;
  const uint32_t ta = cx.tmem + ((uint32_t)(32 * q) << 16) + TM_Z + 32 * kq;
  // dz rows nrow (rows 0-1) and 128 + nrow (rows 2-3), keys 32kq.. in key chunk kq/2
  const uint32_t rowa = cx.sbase + OFF_DZ + (kq >> 1) * DZKC + nrow * 128;
  const uint32_t rowb = rowa + 128 * 128;
  float acc0 = 0.f, acc1 = 0.f, wv0 = 0.f, wv1 = 0.f;
  int zi = 0, i = -1;  // tiles and blocks of one CTA stay far below 2^31
  for (int g = 0;; ++g) {
    const int ms = g % MST;
    if (!WAIT(&B->mfull[ms], (g / MST) & 1)) return;
    const int flags = cx.hdr[ms].flags, c = cx.hdr[ms].c, direct = cx.hdr[ms].direct;
    if (flags & F_FIRST) {
      ++i;
      if (!WAIT(&B->qfull, i & 1)) return;
      wv0 = w_s[nrow];
      wv1 = w_s[128 + nrow];
      acc0 = acc1 = 0.f;
    }
    const float* disb = rec_dis(cx, ms);
#pragma unroll 1
    for (int x = 0; x < 2; ++x) {
      const int r = 2 * x + (q >> 1);
      const float wsc = (x == 0 ? wv0 : wv1) * pow2f(c);
      const uint64_t wsc2 = pack2(__float_as_uint(wsc), __float_as_uint(wsc));
      const float* dr = disb + r * kBM + 32 * kq;
      if (!WAIT(&B->zfull, zi & 1)) return;
      if (tdz == 0) TRACE(x == 0 ? EV_DZ_ZA : EV_DZ_ZB, g);
      tc_fence_after();
      uint32_t pk[16];
      float ad = 0.f;  // direct dW: this tile's sum
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // keys 16hh .. 16hh+15 of the thread's 32
        float z[16];
        tmem_ld16(ta + 16 * hh, z);
        tmem_wait_ld_dep16(z);
        if (hh == 1) {
          tc_fence_before();
          mbar_arrive(&B->zempty);  // the buffer is free for the next Z MMA
        }
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dr + 16 * hh + 4 * j4);
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const float z0 = z[4 * j4 + 2 * e2], z1 = z[4 * j4 + 2 * e2 + 1];
            const float dA = e2 == 0 ? d4.x : d4.z, dB = e2 == 0 ? d4.y : d4.w;
            const uint64_t t2 = mul_f32x2(pack2(__float_as_uint(dA), __float_as_uint(dB)), wsc2);  // dI w 2^c
            const float v0 = z0 > 0.f ? __uint_as_float((uint32_t)t2) : 0.f;
            const float v1 = z1 > 0.f ? __uint_as_float((uint32_t)(t2 >> 32)) : 0.f;
            pk[8 * hh + 2 * j4 + e2] = pack_half2(v0, v1);
            if (direct) ad = fmaf(dA, fmaxf(z0, 0.f), fmaf(dB, fmaxf(z1, 0.f), ad));
          }
        }
      }
      ++zi;
      if (x == 0)
        acc0 += ad;
      else
        acc1 += ad;
      // the dz tile is free once the previous tile's dQ and dK MMAs are complete
      if (x == 0 && !WAIT(&B->dzempty, (g & 1) ^ 1)) return;
      const uint32_t row = x == 0 ? rowa : rowb;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const uint32_t c8 = (kq & 1) * 4 + c4;
        st_shared_v4(row + ((c8 ^ (nrow & 7)) << 4), pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&B->dzfull);
    if (tdz == 0) TRACE(EV_DZ_DONE, g);
    if (flags & F_LAST)
      dz_epilogue(p, cx, cx.hdr[ms].row0, cx.hdr[ms].Rb, c, direct, i, acc0, acc1, wv0, wv1);
    if (flags & F_END) return;
  }
}

// ------------------------------------------------------------ dK group ----
// dK warp w (0..7): TMEM lane quarter qw = w % 4 (32 columns d), entries
// 64*(w/4) .. +63 of the tile in two chunks of 32.
__device__ void dk_role(const BParams& p, const Ctx& cx) {
  const int qw = (threadIdx.x >> 5) & 3;
  const int kg = (threadIdx.x - W_DK0 * 32) >> 7;
  float* stage = reinterpret_cast<float*>(cx.smem + OFF_DKST) + ((threadIdx.x >> 5) - W_DK0) * 512;
  Bars* B = cx.bars;
  for (long long g = 0;; ++g) {
    const int ms = (int)(g % MST);
    if (!WAIT(&B->mfull[ms], (g / MST) & 1)) return;
    const int flags = cx.hdr[ms].flags, c = cx.hdr[ms].c, count = cx.hdr[ms].count, batch = cx.hdr[ms].batch;
    float* base = p.u ? p.u : p.dk + (long long)batch * p.S_k * p.D;
    const int* ids = p.u ? rec_pos(cx, ms) : rec_key(cx, ms);
    if (!WAIT(&B->dkfull, g & 1)) return;
    if (threadIdx.x == W_DK0 * 32) TRACE(EV_DK_FULL, (int)g);
    tc_fence_after();
    const float sc = pow2f(-c);
    const uint32_t ta = cx.tmem + ((uint32_t)(qw * 32) << 16) + TM_DK;
#pragma unroll 1
    for (int ch = kg * 2; ch < kg * 2 + 2; ++ch) {
      if (ch * 32 >= count) break;  // uniform: the remaining entries are padding
      const int nrow = min(32, count - ch * 32);
      if (p.u)
        dk_chunk_tmem<false>(base, ids + ch * 32, ta + ch * 32, nrow, sc, p.D, qw * 32, stage);
      else
        dk_chunk_tmem<true>(base, ids + ch * 32, ta + ch * 32, nrow, sc, p.D, qw * 32, stage);
    }
    tc_fence_before();
    mbar_arrive(&B->dkempty);
    mbar_arrive(&B->mempty[ms]);
    if (threadIdx.x == W_DK0 * 32) TRACE(EV_DK_DONE, (int)g);
    if (flags & F_END) return;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) blk_kernel(const BParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctx cx;
  cx.smem = smem;
  cx.sbase = smem_u32(smem);
  cx.bars = reinterpret_cast<Bars*>(smem + OFF_BARS);
  cx.hdr = reinterpret_cast<Hdr*>(smem + OFF_HDR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  cx.abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    Bars* B = cx.bars;
    for (int i = 0; i < KST; ++i) {
      mbar_init(&B->kfull[i], NGT);
      mbar_init(&B->kempty[i], 1);
    }
    for (int i = 0; i < MST; ++i) {
      mbar_init(&B->mfull[i], 1);
      mbar_init(&B->mempty[i], NDKT);
    }
    for (int i = 0; i < BQ; ++i) {
      mbar_init(&B->bfull[i], 1);
      mbar_init(&B->bempty[i], NQT);
    }
    mbar_init(&B->qfull, NQT);
    mbar_init(&B->qempty, 1);
    mbar_init(&B->zfull, 1);
    mbar_init(&B->zempty, NDZT);
    mbar_init(&B->dzfull, NDZT);
    mbar_init(&B->dzempty, 1);
    mbar_init(&B->dkfull, 1);
    mbar_init(&B->dkempty, NDKT);
    mbar_init(&B->dqfull, 1);
    mbar_init(&B->dqempty, NDZT);
    mbar_init(&B->dwbar, NDZT);
    mbar_init(&B->drain, 2);  // one commit from each MMA issuer
    *cx.abort = 0;
    fence_barrier_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  // everything above overlaps the previous kernel's tail (programmatic
  // dependent launch); the inputs it wrote are read only from here on
  griddep_wait();
  if (threadIdx.x == 0) TRACE_CTA(0, clock64());

  if (warp < W_SCAN) {
    gather_role(p, cx);
  } else if (warp == W_SCAN) {
    scan_role(p, cx);
  } else if (warp == W_MMA) {
    zmma_role(p, cx);  // the whole warp runs the loop; one elected lane issues
  } else if (warp == W_GMMA) {
    gmma_role(p, cx);
  } else if (warp < W_DZ0) {
    q_role(p, cx);
  } else if (warp < W_DK0) {
    dz_role(p, cx);
  } else {
    dk_role(p, cx);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) tmem_dealloc(cx.tmem, TM_COLS);
  if (threadIdx.x == 0) TRACE_CTA(1, clock64());
}

// k (bf16, [B, S_k, D]) -> fp16 [B][S_k + 1][128]: zero padded beyond D, and
// row S_k of each batch zero (padding entries of a tile copy it).
// Launched programmatically after the score-grad kernel (which writes neither
// k nor the workspace), it runs alongside it and waits for it before exiting,
// so that its own completion implies the score-grad's.
__global__ void k_to_f16_kernel(const uint16_t* __restrict__ k, __half* __restrict__ k16, int B, int S_k, int D,
                                unsigned* __restrict__ sched, int nsched) {
  griddep_launch_dependents();  // the next kernel may start its prologue
  if (blockIdx.x == 0 && threadIdx.x < nsched) sched[threadIdx.x] = 0u;  // the following kernels' counters
  const long long rows = (long long)B * (S_k + 1);
  const long long n = rows * (kDP / 8);
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < n;
       x += (long long)gridDim.x * blockDim.x) {
    const int ch = (int)(x % (kDP / 8));
    const long long row = x / (kDP / 8);
    const int b = (int)(row / (S_k + 1));
    const int s = (int)(row % (S_k + 1));
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (s < S_k && ch * 8 < D) val = __ldg(reinterpret_cast<const uint4*>(k + ((long long)b * S_k + s) * D + ch * 8));
    *reinterpret_cast<uint4*>(k16 + row * kDP + ch * 8) =
        make_uint4(bf16x2_to_half2(val.x), bf16x2_to_half2(val.y), bf16x2_to_half2(val.z), bf16x2_to_half2(val.w));
  }
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
// the block's rows are staged in shared memory (rows of up to 2048 slots).
void union_geometry(int S_k, int L, int& W, int& dcap, int& staged) {
  const long long skr = ((long long)S_k + 1023) / 1024 * 1024;
  W = (int)std::min<long long>(skr, L <= 4096 ? 32768 : 4096);
  dcap = std::min(L, W);
  staged = L <= 2048 ? 1 : 0;
}

size_t union_smem_bytes(int W, int dcap, int L, int staged) {
  size_t s = (size_t)10 * (W / 32) * 4 + (size_t)R * dcap * 4;
  if (staged) s += (size_t)2 * R * ((L + 3) & ~3) * 4;
  return std::max<size_t>(s, 2 * NBUCKET * 4);
}

bool set_smem_attr(const void* fn, size_t bytes, std::atomic<int>* done) {
  // per device; raising the attribute twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
  if (done[dev].load(std::memory_order_acquire) >= (int)bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) return false;
  done[dev].store((int)bytes, std::memory_order_release);
  return true;
}

std::atomic<int> g_attr_blk[64];
std::atomic<int> g_attr_union[64];

}  // namespace

cudaError_t launch_k_to_f16(const uint16_t* k, __half* k16, int B, int S_k, int D, unsigned* sched, int nsched,
                            bool pdl, int num_sms, cudaStream_t st) {
  const long long n = (long long)B * (S_k + 1) * (kDP / 8);
  const int blocks = (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, 8LL * num_sms));
  return launch_ex(k_to_f16_kernel, (unsigned)blocks, 256u, 0, st, pdl, k, k16, B, S_k, D, sched, nsched);
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
  if (!dense) {
    const long long ucap = std::min<long long>(S_k, (long long)R * L);
    w.tcap = (int)std::max<long long>(1, (ucap + kBM - 1) / kBM);
    w.rstride = deterministic ? (int)REC_BYTES : REC_POS;
    w.binfo = off;
    off = up(off + (size_t)w.nblocks * 16);
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
    off = up(off + (size_t)w.entries_cap * D * 4);
    if (!dense) {
      w.hist = off;
      off = up(off + (size_t)w.nchunks * S_k * 4);
    }
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
  // programmatic only right after this library's score-grad kernel: the
  // kernel reads k before it waits for its predecessor
  cudaError_t e = launch_k_to_f16(a.k, k16, a.B, a.S_k, a.D, sched, 2, a.after_score_grad != 0, a.num_sms, st);
  if (e != cudaSuccess) return e;
  if (!dense) {
    UParams u{};
    u.idx = a.idx;
    u.dI = a.dI;
    u.w = a.w;
    u.rec = ws + lay.rec;
    u.binfo = reinterpret_cast<int4*>(ws + lay.binfo);
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
    u.ids_global = a.ids_global;
    union_geometry(a.S_k, a.L, u.W, u.dcap, u.staged);
    const size_t sh = union_smem_bytes(u.W, u.dcap, a.L, u.staged);
    // (its static arrays come on top of the dynamic bytes: always raise the limit)
    if (!set_smem_attr((const void*)union_kernel, sh, g_attr_union)) return cudaErrorInvalidValue;
    // it reads the ids before its predecessor completes and dI only after
    e = launch_ex(union_kernel, (unsigned)lay.nblocks, (unsigned)UT, sh, st, true, u);
    if (e != cudaSuccess) return e;
  }
  if (a.deterministic) {
    e = launch_det_sort(a, lay, st);
    if (e != cudaSuccess) return e;
  }
  if (!set_smem_attr((const void*)blk_kernel, SMEM_BYTES, g_attr_blk)) return cudaErrorInvalidValue;
  BParams p{};
  p.q = a.q;
  p.k16 = k16;
  p.w = a.w;
  p.dI = a.dI;
  p.rec = dense ? nullptr : ws + lay.rec;
  p.binfo = dense ? nullptr : reinterpret_cast<const int4*>(ws + lay.binfo);
  p.border = dense ? nullptr : reinterpret_cast<const int*>(ws + lay.border);
  p.dq = a.dq;
  p.dw = a.dw;
  p.dk = a.dk;
  p.u = a.deterministic ? reinterpret_cast<float*>(ws + lay.u) : nullptr;
  p.dq16 = a.dq16;
  p.dw16 = a.dw16;
  p.sched = sched;
  p.status = a.status;
  p.nblocks = lay.nblocks;
  p.wait_ns = 2000000000ull;
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
  e = launch_ex(blk_kernel, (unsigned)grid, (unsigned)NTHREADS, SMEM_BYTES, st, true, p);
  if (e != cudaSuccess) return e;
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

#ifdef IBWD_TRACE
extern "C" __attribute__((visibility("default"))) int ibwd_trace_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace));
}
extern "C" __attribute__((visibility("default"))) int ibwd_trace_poll_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, g_poll_count, bytes < sizeof(g_poll_count) ? bytes : sizeof(g_poll_count));
}
extern "C" __attribute__((visibility("default"))) int ibwd_trace_cta_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, g_trace_cta, bytes < sizeof(g_trace_cta) ? bytes : sizeof(g_trace_cta));
}
#endif

}  // namespace ibwd
