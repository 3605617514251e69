// Gemm stage of the lightning-indexer backward, one query row at a time:
// the kernel behind the allocation-free entry point (indexer_bwd_gemm_noalloc),
// whose only scratch is the fp16 copy of k.  Atomic dK, top-k ids local to
// their batch, fp32 outputs.
//
// Definition (cudnn-frontend #730 "optimize SM100 gradient kernels",
// benchmark-harness comment, ref_grads), per query row t and selected key
// s = idx[t,j] (any id outside [0, S_k) is padding and skipped):
//   z[s,h]  = q[t,h,:] . k[s,:];   dW[t,h] = sum_s dI[t,s] relu(z[s,h])
//   dz[s,h] = dI[t,s] w[t,h] [z[s,h] > 0]
//   dQ[t,h] = sum_s dz[s,h] k[s,:];   dK[s] += sum_h dz[s,h] q[t,h,:]
//
// Design: one persistent CTA per SM walks its query rows (a low-discrepancy
// permutation of all rows, claimed from a counter).  Each row's valid slots
// are compacted into tiles of 128 keys, the M = 128 dimension of every MMA:
//   MMA1  Z^T[128 s, 64 h]   = Ksel[128 s, 128 d] . Q^T          (TMEM, fp32)
//   MMA2  dK^T[128 d, 128 s] = Q^T[128 d, 64 h] . dz^T[64 h, 128 s] (TMEM, fp32)
//   MMA3  dQ^T[128 d, 64 h] += Ksel^T[128 d, 128 s] . dz[128 s, 64 h]
// Operands are fp16 in 128-byte-swizzled shared memory (k converted once, q
// per row, dz with a per-row power-of-two scale 2^c undone in the fp32
// epilogues).  The selected key rows are gathered by 16-byte cp.async; dK
// leaves TMEM transposed (lane = column d) for full-line reductions.
//
// Warp roles (24 warps; a warp reaches TMEM lanes 32*(warp%4) .. +31):
//   0-3   gather, and each row's dQ epilogue (through a staging row and a
//   bulk copy when every row is one tile);  4 scan (row ids and dI
//   staged by bulk copies one row ahead, compaction into tile metadata);
//   5 MMA issuer and TMEM owner;  6-7 Q loader (the row's q by one bulk
//   copy, then fp16 conversion);  8-15 dz (two groups of four for heads
//   0-31 / 32-63: dW partials, fp16 dz tile, dW reduction);  16-23 dK
//   (fp32 red.global.add of the transposed tile rows).
// Every mbarrier wait is bounded: on expiry the kernel raises a status bit,
// all roles unwind, in-flight copies and MMAs are drained and TMEM is freed.
#include <algorithm>
#include <atomic>

#include "kcommon.cuh"

namespace ibwd {
namespace {

constexpr int KST = 2;  // K-tile stages
constexpr int MST = 8;  // tile-metadata ring (deep enough to hide the per-row scan)
constexpr int RQ = 16;  // row-order ring: the scan runs at most ~MST + 2 rows ahead of the Q loader
constexpr int NTHREADS = 768;
constexpr int W_GATHER0 = 0, W_SCAN = 4, W_MMA = 5, W_Q0 = 6, W_DZ0 = 8, W_DK0 = 16;
constexpr int NGT = 128;                  // gather threads
constexpr int NQT = 64;                   // Q-loader threads
constexpr int NDZT = 256;                 // dz threads (two groups of 128)
constexpr int NDKT = 256;                 // dK threads (two groups of 128)

constexpr uint32_t KTILE_BYTES = kBM * kDP * 2;   // 32 KB
constexpr uint32_t KHALF_BYTES = kBM * 64 * 2;    // one 64-column half of a K tile
constexpr uint32_t QTILE_BYTES = kHP * kDP * 2;   // 16 KB
constexpr uint32_t QHALF_BYTES = kHP * 64 * 2;
constexpr uint32_t DZTILE_BYTES = kBM * kHP * 2;  // 16 KB

// TMEM columns: Z double buffer, dK double buffer, dQ double buffer.
constexpr uint32_t TM_Z = 0, TM_DK = 128, TM_DQ = 384, TM_COLS = 512;

struct TileMeta {
  int key[kBM];    // selected key (row of k within the batch)
  float dis[kBM];  // dI[t, j] * 2^c
  int r, count, c, flags;
};
enum { F_FIRST = 1, F_LAST = 2, F_END = 4 };

struct Bars {
  uint64_t kfull[KST], kempty[KST];
  uint64_t mfull[MST], mempty[MST];
  uint64_t rowfull[2];
  uint64_t qfull[2];
  uint64_t qraw[2];
  uint64_t zfull[2], zempty[2];
  uint64_t dzfull[2], dzempty[2];
  uint64_t dkfull[2], dkempty[2];
  uint64_t dqfull[2], dqempty[2];
  uint64_t dwred[2];
  uint64_t rowid[RQ];
  uint64_t dqst_free, dqst_full;  // one-tile rows: the dQ staging row
  uint64_t drain;
};

// Shared-memory layout.  With rows of one tile (kOneTile: L <= 128) a
// staged row takes 1 KB instead of 16 KB, and the room holds a row of dQ
// (fp32 [H][D]) on its way out by one bulk copy.
template <bool kOneTile>
struct Geo {
  static constexpr uint32_t ROW_BYTES = kOneTile ? 1024 : 16384;  // one staged row: idx | dI
  static constexpr uint32_t DQST_BYTES = kOneTile ? kHP * kDP * 4 : 0;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_Q = OFF_K + KST * KTILE_BYTES;
  static constexpr uint32_t OFF_DZ = OFF_Q + 2 * QTILE_BYTES;
  static constexpr uint32_t OFF_QRAW = OFF_DZ + 2 * DZTILE_BYTES;  // two rows of q as they are (bf16 [H][D])
  static constexpr uint32_t OFF_ROW = OFF_QRAW + 2 * QTILE_BYTES;
  static constexpr uint32_t OFF_DQST = OFF_ROW + 2 * ROW_BYTES;
  static constexpr uint32_t OFF_META = OFF_DQST + DQST_BYTES;
  static constexpr uint32_t OFF_W = OFF_META + MST * sizeof(TileMeta);
  static constexpr uint32_t OFF_RED = OFF_W + 2 * kHP * 4;
  static constexpr uint32_t OFF_BARS = OFF_RED + 2 * 4 * kHP * 4;  // [2][4 warps][64 heads]
  static constexpr uint32_t OFF_ROWQ = OFF_BARS + sizeof(Bars);  // int[RQ]: rows in this CTA's order, -1 = end
  static constexpr uint32_t OFF_DKST = (OFF_ROWQ + RQ * 4 + 15) & ~15u;  // dK transpose stages, 2 KB per dK warp
  static constexpr uint32_t OFF_MISC = OFF_DKST + (NDKT / 32) * 16 * 32 * 4;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(OFF_BARS % 8 == 0 && OFF_ROW % 16 == 0, "alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct KParams {
  const uint16_t* q;
  const __half* k16;   // [B][S_k + 1][128]; row S_k of each batch is zero
  const float* w;
  const float* dI;
  const int32_t* idx;
  float* dq;
  float* dw;
  float* dk;
  unsigned* sched;  // row counter in the scratch, zeroed by the k conversion kernel
  unsigned* status;
  long long rows;
  unsigned long long perm_mul;
  unsigned long long wait_ns;
  int B, S_q, S_k, H, D, L;
  int staged;  // rows are staged in shared memory by bulk copies
  const unsigned* select;  // if set: the kernel runs only when *select == 1 (written by an earlier kernel)
};

__device__ __forceinline__ long long row_of(long long u, const KParams& p) {
  return (long long)(((unsigned long long)u * p.perm_mul) % (unsigned long long)p.rows);
}

struct Ctx {
  uint32_t sbase;
  uint8_t* smem;
  TileMeta* meta;
  float* w_s;
  float* red_s;
  Bars* bars;
  volatile int* abort;
  uint32_t tmem;
  int* rowq;
};

// Every role waits with whole, converged warps; the vote makes the outcome
// warp-uniform, so that a wait that gives up in one lane never leaves the
// others of its warp in a warp-collective instruction alone.
#define WAIT(bar, par) __all_sync(0xffffffffu, mbar_wait((bar), (par), cx.abort, p.status, p.wait_ns))
#define WAITW(bar, par) WAIT(bar, par)

// Optional per-tile timeline (clock64 stamps of each role's progress in the
// first CTAs), compiled only with -DIBWD_TRACE for pipeline analysis.
enum RowTraceEv {
  RV_SCAN_PUB, RV_GATHER, RV_Q_START, RV_Q_FREE, RV_Q_DONE, RV_MMA_Z, RV_MMA_DK, RV_MMA_DQ, RV_DZ_START,
  RV_DZ_DONE, RV_EPI_DONE, RV_DW_DONE, RV_DK_START, RV_DK_DONE, RV_COUNT
};
#ifdef IBWD_TRACE
constexpr int RTRACE_CTAS = 4, RTRACE_TILES = 256;
__device__ unsigned long long g_rtrace[RTRACE_CTAS][RV_COUNT][RTRACE_TILES];
#define RTRACE(ev, g)                                                                                       \
  do {                                                                                                      \
    if (blockIdx.x < RTRACE_CTAS && (g) >= 0 && (g) < RTRACE_TILES && (threadIdx.x & 31) == 0)             \
      g_rtrace[blockIdx.x][ev][g] = clock64();                                                              \
  } while (0)
#else
#define RTRACE(ev, g) \
  do {                \
  } while (0)
#endif

// ------------------------------------------------------------ Q loader ----
// A row's q (H*D bf16, contiguous) arrives by one bulk copy into a raw
// buffer, issued a row ahead; the loader threads then convert it into the
// fp16, 128-byte-swizzled Q operand once that buffer is free.  The copy's
// latency stays off the MMA chain.
template <bool kOneTile>
__device__ void q_role(const KParams& p, const Ctx& cx) {
  using G = Geo<kOneTile>;
  const int tid = threadIdx.x - W_Q0 * 32;  // 0..63
  const uint32_t rowq_bytes = (uint32_t)(p.H * p.D * 2);
  long long issued = -1, landed = -1;  // last rows whose raw copy was issued / waited for
  auto issue_raw = [&](long long i, long long r) {
    if (tid == 0) {
      const int b = (int)(i & 1);
      mbar_arrive_expect_tx(&cx.bars->qraw[b], rowq_bytes);
      bulk_g2s(cx.sbase + G::OFF_QRAW + b * QTILE_BYTES, p.q + r * p.H * p.D, rowq_bytes, &cx.bars->qraw[b]);
    }
    issued = i;
  };
  // copies still in flight (at most two) must land before the CTA can exit
  auto drain = [&]() {
    if (tid == 0)
      for (long long j = landed + 1; j <= issued; ++j)
        drain_wait(&cx.bars->qraw[j & 1], (uint32_t)((j >> 1) & 1), p.status, p.wait_ns);
  };
  if (!WAIT(&cx.bars->rowid[0], 0u)) return;
  long long r = cx.rowq[0];
  if (r >= 0) issue_raw(0, r);
  for (long long i = 0; r >= 0; ++i) {
    const int qb = (int)(i & 1);
    // the next row's copy into the other raw buffer, once both loader warps
    // have converted row i - 1 out of it (their qfull arrivals)
    if (!WAIT(&cx.bars->rowid[(i + 1) % RQ], (uint32_t)(((i + 1) / RQ) & 1))) return drain();
    const long long rn = cx.rowq[(i + 1) % RQ];
    if (i >= 1 && !WAIT(&cx.bars->qfull[(i + 1) & 1], (uint32_t)(((i - 1) >> 1) & 1))) return drain();
    if (rn >= 0) issue_raw(i + 1, rn);
    if (tid == 0) RTRACE(RV_Q_START, (int)i);
    const float wv = tid < p.H ? __ldg(p.w + r * p.H + tid) : 0.f;
    if (!WAIT(&cx.bars->qraw[qb], (uint32_t)((i >> 1) & 1))) return drain();
    landed = i;
    // buffer qb was last used by row i-2: all its MMAs and dz reads are done
    // once that row's dQ accumulator is complete
    if (i >= 2 && !WAIT(&cx.bars->dqfull[qb], (uint32_t)(((i - 2) >> 1) & 1))) return drain();
    if (tid == 0) RTRACE(RV_Q_FREE, (int)i);
    const uint8_t* raw = cx.smem + G::OFF_QRAW + qb * QTILE_BYTES;
    const uint32_t qs = cx.sbase + G::OFF_Q + qb * QTILE_BYTES;
    bool bad = false;
#pragma unroll 4
    for (int it = 0; it < 16; ++it) {
      const int x = tid + it * NQT;  // 16-byte chunk: head h, column chunk ch
      const int h = x >> 4, ch = x & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (h < p.H && ch * 8 < p.D) v = *reinterpret_cast<const uint4*>(raw + (h * p.D + ch * 8) * 2);
      const uint32_t dst = qs + (ch >> 3) * QHALF_BYTES + h * 128 + (((ch & 7) ^ (h & 7)) << 4);
      bad |= bf16x2_out_of_fp16(v.x) || bf16x2_out_of_fp16(v.y) || bf16x2_out_of_fp16(v.z) ||
             bf16x2_out_of_fp16(v.w);
      st_shared_v4(dst, bf16x2_to_half2(v.x), bf16x2_to_half2(v.y), bf16x2_to_half2(v.z), bf16x2_to_half2(v.w));
    }
    if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) atomicOr(p.status, DEV_FP16_RANGE);
    cx.w_s[qb * kHP + tid] = wv;
    // the raw buffer's generic reads precede the next copy into it (async)
    fence_proxy_async_smem();
    mbar_arrive(&cx.bars->qfull[qb]);
    if (tid == 0) RTRACE(RV_Q_DONE, (int)i);
    r = rn;
  }
}

// ----------------------------------------------------------------- scan ---
template <bool kOneTile>
__device__ void scan_role(const KParams& p, const Ctx& cx) {
  using G = Geo<kOneTile>;
  const int lane = threadIdx.x & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint8_t* rowbuf = cx.smem + G::OFF_ROW;
  long long staged_wait = -1;  // last row whose bulk copy was issued but not yet waited for
  // The CTA's first row is blockIdx.x (the grid never exceeds the row
  // count); later rows are claimed from the shared counter, so CTAs that run
  // faster take more rows.  Row numbers go through the permutation.
  // A claim is issued at the start of a row and resolved after that row's
  // first pass, so the atomic's round trip overlaps the pass.
  auto claim_issue = [&]() -> unsigned { return lane == 0 ? atomicAdd(p.sched, 1u) : 0u; };
  auto claim_resolve = [&](unsigned pend) -> long long {
    const unsigned v = __shfl_sync(0xffffffffu, pend, 0);
    const long long u = (long long)gridDim.x + v;
    return u < p.rows ? row_of(u, p) : -1;
  };
  // |w| of a row, loaded early (two heads per lane, H <= 64)
  auto w_load = [&](long long r, float& w0, float& w1) {
    w0 = lane < p.H ? __ldg(p.w + r * p.H + lane) : 0.f;
    w1 = lane + 32 < p.H ? __ldg(p.w + r * p.H + lane + 32) : 0.f;
  };
  auto publish_row = [&](long long i, long long r) {
    if (lane == 0) {
      cx.rowq[i % RQ] = (int)r;
      mbar_arrive(&cx.bars->rowid[i % RQ]);
    }
  };
  auto issue_row = [&](long long i, long long r) {
    const int buf = (int)(i & 1);
    if (lane == 0) {
      // this thread's earlier generic reads of the buffer precede the async writes
      fence_proxy_async_smem();
      const uint32_t dst = smem_u32(rowbuf + buf * G::ROW_BYTES);
      const uint32_t stride = (uint32_t)p.L * 4;  // packed: idx | dI
      mbar_arrive_expect_tx(&cx.bars->rowfull[buf], 2 * stride);
      bulk_g2s(dst, p.idx + r * p.L, stride, &cx.bars->rowfull[buf]);
      bulk_g2s(dst + stride, p.dI + r * p.L, stride, &cx.bars->rowfull[buf]);
    }
    staged_wait = i;
  };

  int g = 0;
  long long r_next = row_of(blockIdx.x, p);
  publish_row(0, r_next);
  if (p.staged) issue_row(0, r_next);
  float wn0, wn1;
  w_load(r_next, wn0, wn1);
  for (long long i = 0;; ++i) {
    const long long r = r_next;
    const unsigned pend = claim_issue();
    const float w0 = wn0, w1 = wn1;
    bool last = false;
    const int32_t* idx;
    const float* dI;
    if (p.staged) {
      const int buf = (int)(i & 1);
      if (!WAIT(&cx.bars->rowfull[buf], (uint32_t)((i >> 1) & 1))) goto done;
      staged_wait = -1;
      __syncwarp();
      const uint8_t* rb = rowbuf + buf * G::ROW_BYTES;
      idx = reinterpret_cast<const int32_t*>(rb);
      dI = reinterpret_cast<const float*>(rb + (uint32_t)p.L * 4);
    } else {
      idx = p.idx + r * p.L;
      dI = p.dI + r * p.L;
    }
    {
      // pass 1: number of valid slots and max |dI| over them
      int nv = 0;
      float mx = 0.f;
      if (p.staged) {
        // 16-byte reads of the staged row, four slots per lane (L % 4 == 0)
        const int nq4 = p.L >> 2;
        for (int q = lane; q < nq4; q += 32) {
          const float4 dv = reinterpret_cast<const float4*>(dI)[q];
          const int4 id = reinterpret_cast<const int4*>(idx)[q];
          const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
          const int ii[4] = {id.x, id.y, id.z, id.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if ((unsigned)ii[k] < (unsigned)p.S_k) {
              ++nv;
              mx = fmaxf(mx, fabsf(dd[k]));
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
      } else {
        for (int j0 = 0; j0 < p.L; j0 += 32) {
          const int j = j0 + lane;
          const bool v = j < p.L && (unsigned)idx[j] < (unsigned)p.S_k;
          if (v) mx = fmaxf(mx, fabsf(dI[j]));
          nv += __popc(__ballot_sync(0xffffffffu, v));
        }
      }
      mx = warp_max(mx);
      // the next row: resolve its claim, publish it, start its staging copy
      // and its w loads
      r_next = claim_resolve(pend);
      publish_row(i + 1, r_next);
      last = r_next < 0;
      if (!last) {
        if (p.staged) issue_row(i + 1, r_next);
        w_load(r_next, wn0, wn1);
      }
      // per-row scale 2^c: max |dI w| 2^c lies in [2^13, 2^14), inside fp16 range
      const int c = dz_scale_exponent(mx * warp_max(fmaxf(fabsf(w0), fabsf(w1))));
      const float sc = pow2f(c);
      const int ntiles = max(1, (nv + kBM - 1) / kBM);
      // pass 2: compact the valid slots, in slot order, into tiles of 128
      int jc = 0, skip = 0;
      for (int tt = 0; tt < ntiles; ++tt, ++g) {
        const int ms = g % MST;
        if (!WAIT(&cx.bars->mempty[ms], (uint32_t)(((g / MST) & 1) ^ 1))) goto done;
        TileMeta& M = cx.meta[ms];
        int fill = 0;
        while (fill < kBM && jc < p.L) {
          const int j = jc + lane;
          const int s = j < p.L ? idx[j] : -1;
          const bool v = (unsigned)s < (unsigned)p.S_k;
          const unsigned mask = __ballot_sync(0xffffffffu, v);
          const int tot = __popc(mask);
          const int rank = __popc(mask & lt_mask);
          const int room = kBM - fill;
          if (v && rank >= skip && rank < skip + room) {
            const int pos = fill + rank - skip;
            M.key[pos] = s;
            M.dis[pos] = dI[j] * sc;
          }
          const int taken = min(tot - skip, room);
          fill += taken;
          if (skip + taken < tot) {
            skip += taken;
          } else {
            skip = 0;
            jc += 32;
          }
        }
        if (lane == 0) {
          M.r = (int)r;
          M.count = fill;
          M.c = c;
          M.flags = (tt == 0 ? F_FIRST : 0) | (tt == ntiles - 1 ? F_LAST : 0) |
                    ((tt == ntiles - 1 && last) ? F_END : 0);
        }
        __syncwarp();
        mbar_arrive(&cx.bars->mfull[ms]);
        RTRACE(RV_SCAN_PUB, g);
      }
    }
    __syncwarp();
    if (last) break;
  }
done:
  // a row copy still in flight must land before the CTA can exit
  if (staged_wait >= 0)
    drain_wait(&cx.bars->rowfull[staged_wait & 1], (uint32_t)((staged_wait >> 1) & 1), p.status, p.wait_ns);
}

// ------------------------------------------------------- dQ epilogue ----
// Row `iq` of this CTA (query row r, scale 2^c) leaves its dQ accumulator:
// warp w of the four gather warps reads TMEM lanes 32w .. 32w+31 (the
// columns d of dQ), all 64 heads, and stores dQ[r, h, d] = acc * 2^-c, one
// 128-byte line per head and warp.
__device__ __forceinline__ bool dq_epilogue(const KParams& p, const Ctx& cx, long long iq, int r, int c) {
  const int qw = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  if (!WAIT(&cx.bars->dqfull[iq & 1], (uint32_t)((iq >> 1) & 1))) return false;
  tc_fence_after();
  const uint32_t ta = cx.tmem + ((uint32_t)(qw * 32) << 16) + TM_DQ + (uint32_t)(iq & 1) * 64;
  const float sc = pow2f(-c);
  const int d = qw * 32 + lane;  // TMEM lane = column of dQ
  float* dst = p.dq + (long long)r * p.H * p.D + d;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float v[32];
    tmem_ld32(ta + half * 32, v);
    tmem_wait_ld_dep(v);
    if (half == 1) {
      tc_fence_before();
      mbar_arrive(&cx.bars->dqempty[iq & 1]);
    }
    if (d < p.D) {
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const int hh = half * 32 + h;
        if (hh < p.H) dst[(long long)hh * p.D] = v[h] * sc;
      }
    }
  }
  return true;
}

// The same for one-tile rows: the four warps write the row, scaled, into a
// staging row laid out as dQ[r] is ([H][D] fp32), and one thread sends it
// out by one bulk copy (dq is 16-byte aligned and D a multiple of 8 at every
// entry point, so each row is 16-byte aligned and H*D*4 a multiple of 16).
// `ne` counts this CTA's staged rows (the staging barriers' phases).
template <bool kOneTile>
__device__ __forceinline__ bool dq_epilogue_staged(const KParams& p, const Ctx& cx, long long iq, int r, int c,
                                                   long long ne) {
  using G = Geo<kOneTile>;
  const int x = threadIdx.x - W_GATHER0 * 32, qw = x >> 5, lane = x & 31;
  if (!WAIT(&cx.bars->dqfull[iq & 1], (uint32_t)((iq >> 1) & 1))) return false;
  // the staging row is free once the previous row's bulk copy has read it
  if (x == 0) {
    bulk_wait_read<0>();
    mbar_arrive(&cx.bars->dqst_free);
  }
  if (!WAIT(&cx.bars->dqst_free, (uint32_t)(ne & 1))) return false;
  tc_fence_after();
  const uint32_t ta = cx.tmem + ((uint32_t)(qw * 32) << 16) + TM_DQ + (uint32_t)(iq & 1) * 64;
  const float sc = pow2f(-c);
  const int d = qw * 32 + lane;  // TMEM lane = column of dQ
  float* st = reinterpret_cast<float*>(cx.smem + G::OFF_DQST) + d;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float v[32];
    tmem_ld32(ta + half * 32, v);
    tmem_wait_ld_dep(v);
    if (half == 1) {
      tc_fence_before();
      mbar_arrive(&cx.bars->dqempty[iq & 1]);
    }
    if (d < p.D) {
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const int hh = half * 32 + h;
        if (hh < p.H) st[hh * p.D] = v[h] * sc;
      }
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(&cx.bars->dqst_full);
  bool ok = true;
  if (x == 0) {
    ok = mbar_wait(&cx.bars->dqst_full, (uint32_t)(ne & 1), cx.abort, p.status, p.wait_ns);
    if (ok) {
      bulk_s2g(p.dq + (long long)r * p.H * p.D, cx.sbase + G::OFF_DQST, (uint32_t)(p.H * p.D * 4));
      bulk_commit();
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0);
}

// --------------------------------------------------------------- gather ---
// Thread x copies chunk (x % 16) of rows (x / 16) + 8i, i = 0..15: every warp
// instruction moves two whole 256-byte key rows.  Row r of the tile lands in
// the 128-byte-swizzle layout: half (chunk / 8), XOR (chunk % 8) ^ (r % 8).
// Each thread's copies arrive on the stage barrier when they land.
// The same warps store each row's dQ (through the staging row when every
// row is one tile): once tile g's K stage is free
// again, the dQ MMA of tile g - KST has completed, and if that tile ended its
// row the row's accumulator is complete; its store overlaps tile g's copies.
template <bool kOneTile>
__device__ void gather_role(const KParams& p, const Ctx& cx) {
  using G = Geo<kOneTile>;
  const int x = threadIdx.x - W_GATHER0 * 32;  // 0..127
  const int rsub = x >> 4, ch = x & 15;
  const uint32_t dst_off = (ch >> 3) * KHALF_BYTES + rsub * 128 + (((ch & 7) ^ rsub) << 4);
  // the last KST tiles, oldest first: query row, scale exponent, row-end
  // flag, row number in this CTA
  int hr[KST], hc[KST];
  bool hlast[KST];
  long long hiq[KST];
#pragma unroll
  for (int i = 0; i < KST; ++i) hlast[i] = false;
  long long iq = -1, ne = 0;
  bool ok = true;
  int g = 0;
  // the row's dQ: staged (counting the staged rows) or stored directly
  auto epilogue = [&](long long eiq, int er, int ec) -> bool {
    if constexpr (kOneTile) return dq_epilogue_staged<kOneTile>(p, cx, eiq, er, ec, ne++);
    return dq_epilogue(p, cx, eiq, er, ec);
  };
  for (;; ++g) {
    const int ms = g % MST;
    if (!WAIT(&cx.bars->mfull[ms], (uint32_t)((g / MST) & 1))) { ok = false; break; }
    const TileMeta& M = cx.meta[ms];
    const int count = M.count, flags = M.flags;
    const long long b = M.r / p.S_q;
    if (flags & F_FIRST) ++iq;
    const int st = g % KST;
    if (!WAIT(&cx.bars->kempty[st], (uint32_t)(((g / KST) & 1) ^ 1))) { ok = false; break; }
    const uint32_t kbase = cx.sbase + G::OFF_K + st * KTILE_BYTES + dst_off;
    const __half* kb = p.k16 + b * (p.S_k + 1) * kDP + ch * 8;
    int key[kBM / 8];
#pragma unroll
    for (int i = 0; i < kBM / 8; ++i) {
      const int row = rsub + 8 * i;
      key[i] = row < count ? M.key[row] : p.S_k;  // padding rows copy the zero row
    }
#pragma unroll
    for (int i = 0; i < kBM / 8; ++i) cp_async16(kbase + i * 1024, kb + (long long)key[i] * kDP, 16);
    cp_async_mbar_arrive_noinc(&cx.bars->kfull[st]);
    if (x == 0) RTRACE(RV_GATHER, g);
    // tile g - KST: its row's dQ, if it ended the row (the history is a
    // shift register, so that it stays in registers)
    if (hlast[0]) {
      if (!epilogue(hiq[0], hr[0], hc[0])) { ok = false; break; }
      if (x == 0) RTRACE(RV_EPI_DONE, g - KST);
    }
#pragma unroll
    for (int i = 0; i + 1 < KST; ++i) {
      hr[i] = hr[i + 1];
      hc[i] = hc[i + 1];
      hlast[i] = hlast[i + 1];
      hiq[i] = hiq[i + 1];
    }
    hr[KST - 1] = M.r;
    hc[KST - 1] = M.c;
    hlast[KST - 1] = (flags & F_LAST) != 0;
    hiq[KST - 1] = iq;
    if (flags & F_END) break;
  }
  // the rows of the last KST tiles, in order
  if (ok) {
#pragma unroll
    for (int i = 0; i < KST; ++i)
      if (hlast[i] && !epilogue(hiq[i], hr[i], hc[i])) break;
  }
  // copies in flight must land (or leave) before the CTA can exit
  cp_async_wait_all();
  if (kOneTile && x == 0) bulk_wait<0>();
}

// ------------------------------------------------------------------ MMA ---
constexpr uint32_t ID_Z = idesc_f16_f32(128, 64, 0, 0);    // Z^T = K . Q^T
constexpr uint32_t ID_DKT = idesc_f16_f32(128, 128, 1, 0);  // dK^T = Q^T . dz^T (Q as MN-major A)
constexpr uint32_t ID_DQ = idesc_f16_f32(128, 64, 1, 1);   // dQ^T = K^T . dz (both MN-major)

template <bool kOneTile>
__device__ __forceinline__ void mma_z(const Ctx& cx, int g, int qb) {
  using G = Geo<kOneTile>;
  const uint64_t a0 = sw128_desc(cx.sbase + G::OFF_K + (g % KST) * KTILE_BYTES, 16, 1024);
  const uint64_t b0 = sw128_desc(cx.sbase + G::OFF_Q + qb * QTILE_BYTES, 16, 1024);
  const uint32_t d = cx.tmem + TM_Z + (g & 1) * 64;
#pragma unroll
  for (int k = 0; k < 8; ++k)  // K = D = 128 in steps of 16
    umma_f16_elect(d, a0 + (((k >> 2) * KHALF_BYTES + (k & 3) * 32) >> 4),
                   b0 + (((k >> 2) * QHALF_BYTES + (k & 3) * 32) >> 4), ID_Z, k > 0);
}

template <bool kOneTile>
__device__ __forceinline__ void mma_dk(const Ctx& cx, int g, int qb) {
  using G = Geo<kOneTile>;
  const uint64_t a0 = sw128_desc(cx.sbase + G::OFF_Q + qb * QTILE_BYTES, QHALF_BYTES, 1024);  // Q^T: M = d, MN-major
  const uint64_t b0 = sw128_desc(cx.sbase + G::OFF_DZ + (g & 1) * DZTILE_BYTES, 16, 1024);    // dz^T: N = s, K-major
  const uint32_t d = cx.tmem + TM_DK + (g & 1) * 128;
#pragma unroll
  for (int k = 0; k < 4; ++k)  // K = H = 64 in steps of 16
    umma_f16_elect(d, a0 + ((k * 2048) >> 4), b0 + ((k * 32) >> 4), ID_DKT, k > 0);
}

template <bool kOneTile>
__device__ __forceinline__ void mma_dq(const Ctx& cx, int g, int qd, bool first) {
  using G = Geo<kOneTile>;
  const uint64_t a0 = sw128_desc(cx.sbase + G::OFF_K + (g % KST) * KTILE_BYTES, KHALF_BYTES, 1024);
  const uint64_t b0 = sw128_desc(cx.sbase + G::OFF_DZ + (g & 1) * DZTILE_BYTES, DZTILE_BYTES, 1024);
  const uint32_t d = cx.tmem + TM_DQ + qd * 64;
#pragma unroll
  for (int k = 0; k < 8; ++k)  // K = 128 keys in steps of 16
    umma_f16_elect(d, a0 + ((k * 2048) >> 4), b0 + ((k * 2048) >> 4), ID_DQ, (first && k == 0) ? 0u : 1u);
}

// Tile g's MMAs are dK then dQ; Z of tile g+1 goes into the other Z buffer.
// That Z is issued as soon as its inputs (tile metadata, K tile, the row's
// Q operand, a free Z buffer) are ready: before tile g's dK when they already
// are, so the dz warps find it waiting, else between dK and dQ, else after
// dQ.  So tile g's dQ, and the release of its K stage, dz tile and (for the
// row's last tile) Q buffer behind it, never wait on the next tile's inputs:
// with one-tile rows those inputs are what that release makes room for.
template <bool kOneTile>
__device__ void mma_role(const KParams& p, const Ctx& cx) {
  using G = Geo<kOneTile>;
  Bars* B = cx.bars;
  int g = 0;
  long long iq = 0;
  int flags = 0, nflags = 0;
  long long niq = 0;
  bool zn = false;  // Z of tile g+1 issued
  // Z of tile g1 = g + 1 when its inputs are ready; `block` waits for them,
  // otherwise a test that does not wait.  Returns -1 once a wait gave up.
  auto try_z = [&](bool block) -> int {
    const int g1 = g + 1;
    if (block) {
      if (!WAITW(&B->mfull[g1 % MST], (uint32_t)((g1 / MST) & 1))) return -1;
    } else if (!__all_sync(0xffffffffu, mbar_test(&B->mfull[g1 % MST], (uint32_t)((g1 / MST) & 1)))) {
      return 0;
    }
    const int nf = cx.meta[g1 % MST].flags;
    const long long ni = iq + ((nf & F_FIRST) ? 1 : 0);
    auto ready = [&](uint64_t* bar, uint32_t par) -> int {
      if (block) return WAITW(bar, par) ? 1 : -1;
      return __all_sync(0xffffffffu, mbar_test(bar, par)) ? 1 : 0;
    };
    int st = (nf & F_FIRST) ? ready(&B->qfull[ni & 1], (uint32_t)((ni >> 1) & 1)) : 1;
    if (st == 1) st = ready(&B->kfull[g1 % KST], (uint32_t)((g1 / KST) & 1));
    if (st == 1) st = ready(&B->zempty[g1 & 1], (uint32_t)(((g1 >> 1) & 1) ^ 1));
    if (st != 1) return st;
    // the key tile was written by cp.async (generic proxy): order it before
    // the tensor core's reads
    fence_proxy_async_smem();
    tc_fence_after();
    mma_z<kOneTile>(cx, g1, (int)(ni & 1));
    umma_commit_elect(&B->zfull[g1 & 1]);
    RTRACE(RV_MMA_Z, g1);
    nflags = nf;
    niq = ni;
    zn = true;
    return 1;
  };
  if (!WAITW(&B->mfull[0], 0)) goto drain;
  flags = cx.meta[0].flags;
  if (!WAITW(&B->qfull[0], 0) || !WAITW(&B->kfull[0], 0)) goto drain;
  fence_proxy_async_smem();
  tc_fence_after();
  mma_z<kOneTile>(cx, 0, 0);
  umma_commit_elect(&B->zfull[0]);
  RTRACE(RV_MMA_Z, 0);
  for (;;) {
    const bool more = !(flags & F_END);
    if (more && try_z(false) < 0) goto drain;
    if (!WAITW(&B->dzfull[g & 1], (uint32_t)((g >> 1) & 1))) goto drain;
    if (!WAITW(&B->dkempty[g & 1], (uint32_t)(((g >> 1) & 1) ^ 1))) goto drain;
    tc_fence_after();
    mma_dk<kOneTile>(cx, g, (int)(iq & 1));
    umma_commit_elect(&B->dkfull[g & 1]);
    RTRACE(RV_MMA_DK, g);
    if (more && !zn && try_z(false) < 0) goto drain;
    if ((flags & F_FIRST) && !WAITW(&B->dqempty[iq & 1], (uint32_t)(((iq >> 1) & 1) ^ 1))) goto drain;
    tc_fence_after();
    mma_dq<kOneTile>(cx, g, (int)(iq & 1), (flags & F_FIRST) != 0);
    RTRACE(RV_MMA_DQ, g);
    umma_commit_elect(&B->kempty[g % KST]);
    umma_commit_elect(&B->dzempty[g & 1]);
    if (flags & F_LAST) umma_commit_elect(&B->dqfull[iq & 1]);
    if (!more) break;
    if (!zn && try_z(true) < 0) goto drain;
    ++g;
    flags = nflags;
    iq = niq;
    zn = false;
  }
drain:
  // every MMA issued so far completes before TMEM can be released
  __syncwarp();
  umma_commit_elect(&B->drain);
  drain_wait(&B->drain, 0, p.status, p.wait_ns);
}

// ------------------------------------------------------------ dz group ----
// Group `hg` (0 or 1) owns heads 32*hg .. 32*hg+31 of every tile row.
template <bool kOneTile>
__device__ void dz_role(const KParams& p, const Ctx& cx) {
  using G = Geo<kOneTile>;
  const int qw = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int s = qw * 32 + lane;  // tile row = TMEM lane
  const int tdz = threadIdx.x - W_DZ0 * 32;  // 0..255
  const int hg = tdz >> 7;                    // head group
  float acc[32];
#pragma unroll
  for (int h = 0; h < 32; ++h) acc[h] = 0.f;
  long long iq = -1;
  for (int g = 0;; ++g) {
    const int ms = g % MST;
    if (!WAIT(&cx.bars->mfull[ms], (uint32_t)((g / MST) & 1))) break;
    const TileMeta& M = cx.meta[ms];
    const int flags = M.flags, count = M.count, c = M.c, r = M.r;
    if (flags & F_FIRST) {
      ++iq;
#pragma unroll
      for (int h = 0; h < 32; ++h) acc[h] = 0.f;
      if (!WAIT(&cx.bars->qfull[iq & 1], (uint32_t)((iq >> 1) & 1))) break;
    }
    const float dis = s < count ? M.dis[s] : 0.f;
    // dI 2^c w for this row's 32 heads, as fp32 pairs
    const uint64_t* w2 = reinterpret_cast<const uint64_t*>(cx.w_s + (iq & 1) * kHP + hg * 32);
    const uint64_t dis2 = pack2(__float_as_uint(dis), __float_as_uint(dis));
    if (!WAIT(&cx.bars->zfull[g & 1], (uint32_t)((g >> 1) & 1))) break;
    if (!WAIT(&cx.bars->dzempty[g & 1], (uint32_t)(((g >> 1) & 1) ^ 1))) break;
    tc_fence_after();
    if (tdz == 0) RTRACE(RV_DZ_START, g);
    const uint32_t za = cx.tmem + ((uint32_t)(qw * 32) << 16) + TM_Z + (uint32_t)(g & 1) * 64 + hg * 32;
    const uint32_t dzrow = cx.sbase + G::OFF_DZ + (g & 1) * DZTILE_BYTES + s * 128;
#pragma unroll
    for (int zh = 0; zh < 2; ++zh) {
      float z[16];
      tmem_ld16(za + zh * 16, z);
      tmem_wait_ld_dep16(z);
      if (zh == 1) {
        tc_fence_before();
        mbar_arrive(&cx.bars->zempty[g & 1]);
      }
#pragma unroll
      for (int c8 = zh * 2; c8 < zh * 2 + 2; ++c8) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h0 = c8 * 8 + e * 2;
          const float z0 = z[h0 - zh * 16], z1 = z[h0 + 1 - zh * 16];
          const uint64_t dw = mul_f32x2(dis2, w2[h0 >> 1]);
          const bool p0 = z0 > 0.f, p1 = z1 > 0.f;
          if (p0) acc[h0] = fmaf(dis, z0, acc[h0]);
          if (p1) acc[h0 + 1] = fmaf(dis, z1, acc[h0 + 1]);
          const float d0 = p0 ? __uint_as_float((uint32_t)dw) : 0.f;
          const float d1 = p1 ? __uint_as_float((uint32_t)(dw >> 32)) : 0.f;
          pk[e] = pack_half2(d0, d1);
        }
        const int chunk = hg * 4 + c8;  // 16-byte chunk of the 128-byte dz row
        st_shared_v4(dzrow + ((chunk ^ (s & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&cx.bars->dzfull[g & 1]);
    if (tdz == 0) RTRACE(RV_DZ_DONE, g);
    if (flags & F_LAST) {
      // dW[t,h] = 2^-c sum over the 128 tile rows of acc[h]: a butterfly
      // leaves head 32*hg + lane summed over the warp, then the four warps'
      // partials are added in a fixed order
#pragma unroll
      for (int step = 0; step < 5; ++step) {
        const int o = 16 >> step, n = 16 >> step;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < n; ++k) {
          const float send = upper ? acc[k] : acc[k + n];
          const float keep = upper ? acc[k + n] : acc[k];
          acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      float* red = cx.red_s + (iq & 1) * 4 * kHP;
      red[qw * kHP + hg * 32 + lane] = acc[0];
      mbar_arrive(&cx.bars->dwred[iq & 1]);
      if (tdz < kHP) {
        if (!WAIT(&cx.bars->dwred[iq & 1], (uint32_t)((iq >> 1) & 1))) break;
        if (tdz < p.H)
          p.dw[(long long)r * p.H + tdz] =
              (((red[tdz] + red[kHP + tdz]) + red[2 * kHP + tdz]) + red[3 * kHP + tdz]) * pow2f(-c);
      }
      if (tdz == 0) RTRACE(RV_DW_DONE, g);
    }
    if (flags & F_END) break;
  }
}

// ------------------------------------------------------------ dK group ----
// TMEM holds dK^T: lane = column d, TMEM column = tile row.  Group kg owns
// tile rows 64*kg .. 64*kg+63 in two chunks of 32.
template <bool kOneTile>
__device__ void dk_role(const KParams& p, const Ctx& cx) {
  using G = Geo<kOneTile>;
  const int qw = (threadIdx.x >> 5) & 3;
  const int kg = (threadIdx.x - W_DK0 * 32) >> 7;
  float* stage = reinterpret_cast<float*>(cx.smem + G::OFF_DKST) + ((threadIdx.x >> 5) - W_DK0) * (16 * 32);
  for (int g = 0;; ++g) {
    const int ms = g % MST;
    if (!WAIT(&cx.bars->mfull[ms], (uint32_t)((g / MST) & 1))) return;
    const TileMeta& M = cx.meta[ms];
    const int flags = M.flags, c = M.c, r = M.r, count = M.count;
    float* base = p.dk + (long long)(r / p.S_q) * p.S_k * p.D;
    if (!WAIT(&cx.bars->dkfull[g & 1], (uint32_t)((g >> 1) & 1))) return;
    tc_fence_after();
    if (threadIdx.x == W_DK0 * 32) RTRACE(RV_DK_START, g);
    const float sc = pow2f(-c);
    const uint32_t ta = cx.tmem + ((uint32_t)(qw * 32) << 16) + TM_DK + (uint32_t)(g & 1) * 128;
#pragma unroll 1
    for (int ch = kg * 2; ch < kg * 2 + 2; ++ch) {
      if (ch * 32 >= count) break;  // uniform: the remaining rows are padding
      float v[32];
      tmem_ld32(ta + ch * 32, v);
      tmem_wait_ld_dep(v);
      dk_chunk<true>(base, M.key + ch * 32, v, min(32, count - ch * 32), sc, p.D, qw * 32, stage);
    }
    tc_fence_before();
    mbar_arrive(&cx.bars->dkempty[g & 1]);
    mbar_arrive(&cx.bars->mempty[ms]);
    if (threadIdx.x == W_DK0 * 32) RTRACE(RV_DK_DONE, g);
    if (flags & F_END) return;
  }
}

template <bool kOneTile>
__global__ void __launch_bounds__(NTHREADS, 1) gemm_rows_kernel(const KParams p) {
  if (p.select != nullptr) {
    // the choice was made on the device: the blocked kernel before never
    // lets this one launch early, so the wait costs nothing, and a call that
    // kernel served leaves before any setup
    griddep_wait();
    if (__ldcg(p.select) != 1u) return;
  }
  using G = Geo<kOneTile>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctx cx;
  cx.smem = smem;
  cx.sbase = smem_u32(smem);
  cx.meta = reinterpret_cast<TileMeta*>(smem + G::OFF_META);
  cx.w_s = reinterpret_cast<float*>(smem + G::OFF_W);
  cx.red_s = reinterpret_cast<float*>(smem + G::OFF_RED);
  cx.bars = reinterpret_cast<Bars*>(smem + G::OFF_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::OFF_MISC);
  cx.abort = reinterpret_cast<volatile int*>(smem + G::OFF_MISC + 4);
  cx.rowq = reinterpret_cast<int*>(smem + G::OFF_ROWQ);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    Bars* B = cx.bars;
    for (int i = 0; i < KST; ++i) {
      mbar_init(&B->kfull[i], NGT);
      mbar_init(&B->kempty[i], 1);
    }
    for (int i = 0; i < MST; ++i) {
      mbar_init(&B->mfull[i], 32);
      mbar_init(&B->mempty[i], NDKT);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->rowfull[i], 1);
      mbar_init(&B->qfull[i], NQT);
      mbar_init(&B->qraw[i], 1);
      mbar_init(&B->zfull[i], 1);
      mbar_init(&B->zempty[i], NDZT);
      mbar_init(&B->dzfull[i], NDZT);
      mbar_init(&B->dzempty[i], 1);
      mbar_init(&B->dkfull[i], 1);
      mbar_init(&B->dkempty[i], NDKT);
      mbar_init(&B->dqfull[i], 1);
      mbar_init(&B->dqempty[i], NGT);
      mbar_init(&B->dwred[i], NDZT);
    }
    for (int i = 0; i < RQ; ++i) mbar_init(&B->rowid[i], 1);
    mbar_init(&B->dqst_free, 1);
    mbar_init(&B->dqst_full, NGT);
    mbar_init(&B->drain, 1);
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
  griddep_wait();  // the fp16 copy of k is written by the kernel before

  if (warp < W_SCAN) {
    gather_role<kOneTile>(p, cx);
  } else if (warp == W_SCAN) {
    scan_role<kOneTile>(p, cx);
  } else if (warp == W_MMA) {
    mma_role<kOneTile>(p, cx);  // the whole warp runs the loop; one elected lane issues
  } else if (warp < W_DZ0) {
    q_role<kOneTile>(p, cx);
  } else if (warp < W_DK0) {
    dz_role<kOneTile>(p, cx);
  } else {
    dk_role<kOneTile>(p, cx);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) tmem_dealloc(cx.tmem, TM_COLS);
}

unsigned long long gcd_u64(unsigned long long a, unsigned long long b) {
  while (b) {
    unsigned long long t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Multiplier of the row permutation u -> u*A mod rows: the golden-ratio
// point of rows, nudged to be coprime with rows (a bijection).
unsigned long long row_permutation_multiplier(long long rows) {
  if (rows <= 2) return 1;
  unsigned long long a = (unsigned long long)((double)rows * 0.6180339887498949);
  if (a < 1) a = 1;
  while (gcd_u64(a, (unsigned long long)rows) != 1) ++a;
  return a % (unsigned long long)rows;
}

std::atomic<bool> g_attr_rows[64];

}  // namespace

// Scratch of the per-row kernel: its row counter (one 256-byte block), then
// the fp16 copy of k, 256 bytes per key row plus one zero row per batch.
size_t rows_workspace_bytes(int B, int S_k) { return 256 + (size_t)B * ((size_t)S_k + 1) * kDP * 2; }

cudaError_t prepare_gemm_rows() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && g_attr_rows[dev].load(std::memory_order_acquire)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_rows_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Geo<false>::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<true>::SMEM_BYTES);
  if (e == cudaSuccess && dev >= 0 && dev < 64) g_attr_rows[dev].store(true, std::memory_order_release);
  return e;
}

cudaError_t launch_gemm_rows(const GemmArgs& a, cudaStream_t st) {
  char* ws = static_cast<char*>(a.ws);
  unsigned* sched = reinterpret_cast<unsigned*>(ws);
  __half* k16 = reinterpret_cast<__half*>(ws + 256);
  cudaError_t e = launch_k_to_f16(a.k, k16, a.B, a.S_k, a.D, sched, 1, a.status, false, a.num_sms, st);
  if (e != cudaSuccess) return e;
  return launch_gemm_rows_kernel(a, k16, sched, nullptr, st);
}

cudaError_t launch_gemm_rows_kernel(const GemmArgs& a, const __half* k16, unsigned* counter, const unsigned* select,
                                    cudaStream_t st) {
  cudaError_t e = prepare_gemm_rows();
  if (e != cudaSuccess) return e;
  unsigned* sched = counter;
  KParams p{};
  p.q = a.q;
  p.k16 = k16;
  p.w = a.w;
  p.dI = a.dI;
  p.idx = a.idx;
  p.dq = a.dq;
  p.dw = a.dw;
  p.dk = a.dk;
  p.sched = sched;
  p.status = a.status;
  p.rows = (long long)a.B * a.S_q;
  p.perm_mul = row_permutation_multiplier(p.rows);
  p.wait_ns = 2000000000ull;
  p.B = a.B;
  p.S_q = a.S_q;
  p.S_k = a.S_k;
  p.H = a.H;
  p.D = a.D;
  p.L = a.L;
  // rows are staged in shared memory when they fit and are 16-byte aligned
  const bool one_tile = a.L <= kBM;
  p.staged = 2 * (size_t)a.L * 4 <= (one_tile ? Geo<true>::ROW_BYTES : Geo<false>::ROW_BYTES) && a.L % 4 == 0 &&
             (uintptr_t)a.dI % 16 == 0 &&
             (uintptr_t)a.idx % 16 == 0;
  p.select = select;
  const int grid = (int)std::min<long long>(a.num_sms, p.rows);
  // rows of at most 128 slots are one tile each: the dz warps store their dQ
  if (one_tile)
    return launch_ex(gemm_rows_kernel<true>, (unsigned)grid, (unsigned)NTHREADS, Geo<true>::SMEM_BYTES, st, true, p);
  return launch_ex(gemm_rows_kernel<false>, (unsigned)grid, (unsigned)NTHREADS, Geo<false>::SMEM_BYTES, st, true, p);
}

#ifdef IBWD_TRACE
extern "C" __attribute__((visibility("default"))) int ibwd_rtrace_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, g_rtrace, bytes < sizeof(g_rtrace) ? bytes : sizeof(g_rtrace));
}
#endif

}  // namespace ibwd
