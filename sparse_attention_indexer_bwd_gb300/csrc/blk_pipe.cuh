// The blocked gemm kernel (kernel 2 of the lightning-indexer backward, one
// CTA per SM walking blocks of four query rows).  Included once per pair of
// pipeline depths by a translation unit that first defines IBWD_PIPE_KST (K
// tile stages) and IBWD_PIPE_MST (tile-record slots), and IBWD_PIPE_PRIMARY
// for the production pair; everything here is local to that unit except its
// launch_blk_pipe<KST, MST>.
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
//   5-7   Q loader: the block's q rows by two TMA tile loads (bf16, landing
//         in the operand's swizzled layout), converted to fp16 in place; w
//   8-23  dz: Z -> mask, dW partial, fp16 dz tile; at block end dW and the
//         dQ epilogue (TMEM -> fp32)
//   24-31 dK: dK^T tile from TMEM -> fp32 red.global.add (one 128-byte line
//         per warp-instruction lane group) into dk, or plain stores of the
//         entry's row into u at its sorted position (deterministic mode)
// Every mbarrier wait is bounded: on expiry the kernel raises a status bit,
// all roles unwind, in-flight copies and MMAs are drained and TMEM is freed.
#include <atomic>

#include "blk.h"

namespace ibwd {
namespace {
using namespace blk;

// ----------------------------------------------------------- gemm kernel --
constexpr int KST = IBWD_PIPE_KST;  // K-tile stages
constexpr int MST = IBWD_PIPE_MST;  // tile-record ring
constexpr int BQ = 4;   // block ring (scan -> Q loader)
constexpr int NTHREADS = 1024;
constexpr int W_GATHER0 = 0, W_SCAN = 2, W_MMA = 3, W_GMMA = 4, W_Q0 = 5, W_DZ0 = 8, W_DK0 = 24;
constexpr int NGT = 64, NQT = 96, NDZT = 512, NDKT = 256;
constexpr int NKQ = 4;  // key quarters of a tile: four dz warps per TMEM lane quarter

constexpr uint32_t KTILE = kBM * kDP * 2;  // 32 KB: [2 d-halves][128 keys][128 B]
constexpr uint32_t KHALF = kBM * 128;      // 16 KB
constexpr uint32_t QDH = QIMG_HALF;        // Q block, one 64-d half: [256 (r,h)][128 B] = 32 KB
constexpr uint32_t DZKC = NR * 128;        // dz tile, one 64-key chunk: [256 (r,h)][128 B] = 32 KB

constexpr uint32_t TM_Z = 0, TM_DK = 128, TM_DQ = 256, TM_COLS = 512;

enum { F_FIRST = 1, F_LAST = 2, F_END = 4 };

struct Hdr {        // per tile, written by the scan
  int row0;         // global row index of the block's first row
  int Rb;           // rows in the block (1..4)
  int count;        // entries in the tile (the rest are padding)
  int c;            // dz scale exponent of the block
  int flags;
  int batch;
  int qe;           // deterministic mode: max |q| of the block < 2^qe
  int pad;
};

struct Bars {
  uint64_t kfull[KST], kempty[KST];
  uint64_t mfull[MST], mempty[MST];
  uint64_t bfull[BQ], bempty[BQ];
  uint64_t qfull[2], qempty, qraw;  // qfull[h]: (r,h) rows 128h .. 128h+127 of Q converted
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

// Every role waits with whole, converged warps; the vote makes the outcome
// warp-uniform, so that a wait that gives up (timeout or abort) in one lane
// never leaves the others of its warp in a warp-collective instruction
// (tcgen05.ld, shuffles, elect.sync) alone.
#define WAIT(bar, par) __all_sync(FULL, mbar_wait((bar), (uint32_t)(par), cx.abort, p.status, p.wait_ns))
#define WAITW(bar, par) WAIT(bar, par)

// Optional per-tile timeline (clock64 stamps of each role's progress in the
// first CTAs), compiled only with -DIBWD_TRACE for pipeline analysis.
enum TraceEv {
  EV_SCAN_PUB, EV_GATHER_ISSUED, EV_MMA_ZA, EV_MMA_ZB, EV_MMA_DQ, EV_MMA_DK, EV_DZ_ZA, EV_DZ_ZB, EV_DZ_DONE,
  EV_DK_FULL, EV_DK_DONE, EV_Q_START, EV_Q_DONE, EV_EPI_A, EV_EPI_B, EV_EPI_C, EV_COUNT
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
  if (p.test_stall) return;    // nothing issued: the other roles' waits run out
  // Before an early return: the record copies still in flight (the last MST
  // issued, one per ring slot) land before the CTA may exit.
  auto drain_records = [&]() {
    if (!p.dense && lane == 0)
      for (long long j = g > MST ? g - MST : 0; j < g; ++j)
        drain_wait(&B->mfull[j % MST], (uint32_t)((j / MST) & 1), p.status, p.drain_ns);
  };
  for (;; ++i) {
    const long long b = p.dense ? dense_block_at(p, pos) : (long long)__ldg(p.border + pos);
    const int batch = (int)(b / p.nbpb), jb = (int)(b % p.nbpb);
    const int t0 = jb * R;
    const int Rb = min(R, p.S_q - t0);
    const int row0 = batch * p.S_q + t0;
    // tiles, dz scale exponent and entries of the block (the union pass or the
    // dense scale pass)
    const int4 bi = __ldg(p.binfo + b);
    const int ntiles = bi.x, c = bi.y, U = bi.z;
    const int qe = 0;  // deterministic rows take the block's q exponent from the Q loader
    // publish the block to the Q loader; warm L2 with its q rows
    if (!WAIT(&B->bempty[i % BQ], ((i / BQ) & 1) ^ 1)) return drain_records();
    if (lane == 0) {
      bq[i % BQ] = make_int4(row0, Rb, (int)b, 0);
      mbar_arrive(&B->bfull[i % BQ]);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.q + (long long)row0 * p.H * p.D),
                   "r"((uint32_t)(Rb * p.H * p.D * 2))
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
      if (!WAIT(&B->mempty[ms], ((g / MST) & 1) ^ 1)) return drain_records();
      const int count = min(kBM, U - k * kBM);
      const int flags = (k == 0 ? F_FIRST : 0) | (k == ntiles - 1 ? F_LAST : 0) | (last_blk ? F_END : 0);
      uint8_t* rs = cx.smem + OFF_REC + ms * REC_BYTES;
      if (!p.dense) {
        if (lane == 0) {
          cx.hdr[ms] = Hdr{row0, Rb, max(count, 0), c, flags, batch, qe, 0};
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
          cx.hdr[ms] = Hdr{row0, Rb, count, c, flags, batch, qe, 0};
          mbar_arrive(&B->mfull[ms]);
        }
      }
    }
    if (last_blk) break;
    pos = next;
  }
  // end of the block list for the Q loader
  ++i;
  if (!WAIT(&B->bempty[i % BQ], ((i / BQ) & 1) ^ 1)) return drain_records();
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
      // padding entries hold the zero row S_k; the clamp keeps every address
      // inside k16 whatever a record holds
      const int k0 = min((unsigned)keys[rsub + 8 * i2], (unsigned)p.S_k);
      const int k1 = min((unsigned)keys[rsub + 4 + 8 * i2], (unsigned)p.S_k);
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
// Once the previous block's last MMA that reads Q is complete, the block's q
// rows arrive as two TMA tile loads (the two 64-column halves: 4 rows x 64
// heads x 64 columns of bf16 each, rows past S_q, heads past H and columns
// past D zero), already in the Q operand's swizzled layout; the loader warps
// then convert them to fp16 in place (the range check and, in deterministic
// mode, the block's largest |q| on the way) and put the block's w in shared
// memory.
__device__ void q_role(const BParams& p, const Ctx& cx, const CUtensorMap* qmap) {
  const int tid = threadIdx.x - W_Q0 * 32;  // 0..95
  Bars* B = cx.bars;
  const int4* bq = reinterpret_cast<const int4*>(cx.smem + OFF_BQ);
  float* w_s = reinterpret_cast<float*>(cx.smem + OFF_W);
  unsigned* qmax_s = reinterpret_cast<unsigned*>(cx.smem + OFF_MISC + 8);  // [2]: by block parity
  long long issued = -1, landed = -1;  // the last blocks whose loads were issued / waited for
  // before the role returns: loads in flight have landed
  auto drain = [&]() {
    if (tid == 0 && issued > landed) drain_wait(&B->qraw, (uint32_t)(issued & 1), p.status, p.drain_ns);
  };
  constexpr int ILP = 4;                       // chunks loaded before any is stored
  for (long long i = 0;; ++i) {
    if (!WAIT(&B->bfull[i % BQ], (i / BQ) & 1)) return drain();
    const int row0 = bq[i % BQ].x, Rb = bq[i % BQ].y;
    mbar_arrive(&B->bempty[i % BQ]);
    if (row0 < 0) return drain();
    float wv[(NR + NQT - 1) / NQT];  // w of the block
#pragma unroll
    for (int k = 0; k < (NR + NQT - 1) / NQT; ++k) {
      const int e = tid + NQT * k, r = e >> 6, h = e & 63;
      wv[k] = (e < NR && r < Rb && h < p.H) ? __ldg(p.w + (long long)(row0 + r) * p.H + h) : 0.f;
    }
    // the previous block's last MMAs that read Q (and its w) are complete
    if (!WAIT(&B->qempty, (i & 1) ^ 1)) return drain();
    if (tid == 0) {
      TRACE(EV_Q_START, (int)i);
      if (p.u) qmax_s[i & 1] = 0u;
      const int batch = row0 / p.S_q, t0 = row0 - batch * p.S_q;
      mbar_arrive_expect_tx(&B->qraw, QIMG_BYTES);
      tma_load_4d(cx.sbase + OFF_Q, qmap, 0, 0, t0, batch, &B->qraw);
      tma_load_4d(cx.sbase + OFF_Q + QDH, qmap, 64, 0, t0, batch, &B->qraw);
    }
    issued = i;
#pragma unroll
    for (int k = 0; k < (NR + NQT - 1) / NQT; ++k)
      if (tid + NQT * k < NR) w_s[tid + NQT * k] = wv[k];
    if (!WAIT(&B->qraw, i & 1)) return drain();
    landed = i;
    // rows 0-1 first ((r,h) 0..127 of both 64-column halves: the first Z
    // MMA of the block needs only them), then rows 2-3
    uint32_t mx2 = 0u;  // largest |q| as bf16 bits, per 16-bit lane of a word
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      constexpr int HCH = (int)(QIMG_BYTES / 32);  // chunks of one pair of rows: 2048
      const uint32_t base = cx.sbase + OFF_Q + (uint32_t)hf * (QDH / 2);
#pragma unroll 1
      for (int y0 = tid; y0 < HCH; y0 += ILP * NQT) {
        uint4 v[ILP];
        uint32_t at[ILP];
#pragma unroll
        for (int k = 0; k < ILP; ++k) {
          const int y = y0 + k * NQT;  // chunk y & 1023 of 64-column half y >> 10
          at[k] = base + (uint32_t)(y >> 10) * QDH + (uint32_t)(y & 1023) * 16;
          v[k] = y < HCH ? ld_shared_v4(at[k]) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < ILP; ++k) {
          if (y0 + k * NQT >= HCH) break;
          mx2 = max_u16x2(mx2, max_u16x2(max_u16x2(v[k].x & 0x7FFF7FFFu, v[k].y & 0x7FFF7FFFu),
                                         max_u16x2(v[k].z & 0x7FFF7FFFu, v[k].w & 0x7FFF7FFFu)));
          st_shared_v4(at[k], bf16x2_to_half2(v[k].x), bf16x2_to_half2(v[k].y), bf16x2_to_half2(v[k].z),
                       bf16x2_to_half2(v[k].w));
        }
      }
      if (hf == 1) {
        // above 0x477F: outside the fp16 range
        const unsigned mx = max(mx2 & 0xFFFFu, mx2 >> 16);
        if (__any_sync(FULL, mx > 0x477Fu) && (tid & 31) == 0) atomicOr(p.status, DEV_FP16_RANGE);
        if (p.u) {
          const unsigned m = __reduce_max_sync(FULL, mx);
          if ((tid & 31) == 0 && m != 0u) atomicMax(&qmax_s[i & 1], m);
        }
      }
      // the generic-proxy writes precede the tensor core's reads
      fence_proxy_async_smem();
      mbar_arrive(&B->qfull[hf]);
    }
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
    if (!WAITW(&B->kfull[st], (g / KST) & 1)) break;
    bool ok = true;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      // a block's first Z of each pair of rows waits for those rows' q
      if (((flags & F_FIRST) && !WAITW(&B->qfull[half], i & 1)) || !WAITW(&B->zempty, (zi & 1) ^ 1)) {
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
  drain_wait(&B->drain, 0, p.status, p.drain_ns);
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
  drain_wait(&B->drain, 0, p.status, p.drain_ns);
}

// ------------------------------------------------------------- dz group ---
// dz warp w (0..15): TMEM lane quarter q = w % 4, key quarter kq = w / 4.  For
// each Z buffer (rows 0-1, then rows 2-3) a thread owns the (r,h) row
// 32q + lane of it and the 32 keys 32kq .. 32kq+31 of every tile: it loads
// their z (16 at a time), releases the buffer after the second load, and
// writes dz = dI w 2^c [z > 0] (fp16) into its 64 bytes of the dz row.
//
// dW = sum_s dI relu(z): each thread sums dI relu(z) over its 32 keys of a
// tile as it forms dz (two FMAs per pair of keys, no shared memory), over the
// block's tiles in registers; at block end the four key quarters' partials
// are added in a fixed order.
__device__ void dz_epilogue(const BParams& p, const Ctx& cx, int row0, int Rb, int c, int i, float acc0,
                            float acc1) {
  const int dzw = (threadIdx.x >> 5) - W_DZ0, q = (threadIdx.x >> 5) & 3, kq = dzw >> 2, lane = threadIdx.x & 31;
  const int tdz = threadIdx.x - W_DZ0 * 32;
  float* dwp = reinterpret_cast<float*>(cx.smem + OFF_DWP);
  dwp[kq * NR + 32 * q + lane] = acc0;
  dwp[kq * NR + 128 + 32 * q + lane] = acc1;
  if (!WAIT(&cx.bars->dqfull, i & 1)) return;
  if (tdz == 0) TRACE(EV_EPI_A, i);
  tc_fence_after();
  const int d = 32 * q + lane;  // TMEM lane = column of dQ
  const float sc = pow2f(-c) * p.sm_scale;  // a power of two times s: exact while it stays normal
  const int r = kq;             // dQ columns 64kq .. 64kq+63: the heads of row kq
  const bool ok = r < Rb && d < p.D;
#pragma unroll 1
  for (int cp = 0; cp < 2; ++cp) {  // two 16-column loads in flight at a time
    float v[2][16];
    const uint32_t ta = cx.tmem + ((uint32_t)(32 * q) << 16) + TM_DQ + 64 * kq + 32 * cp;
    tmem_ld16(ta, v[0]);
    tmem_ld16(ta + 16, v[1]);
    tmem_wait_ld_dep16(v[0]);
    tmem_wait_ld_dep16(v[1]);
    if (cp == 1) {
      tc_fence_before();
      mbar_arrive(&cx.bars->dqempty);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int h0 = 32 * cp + 16 * u;
      const long long e0 = ((long long)(row0 + r) * p.H + h0) * p.D + d;
      if (ok) {
        if (p.dq16) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (h0 + j < p.H) p.dq16[e0 + (long long)j * p.D] = to_bf16(v[u][j] * sc);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (h0 + j < p.H) p.dq[e0 + (long long)j * p.D] = v[u][j] * sc;
        }
      }
    }
  }
  mbar_arrive(&cx.bars->dwbar);
  if (tdz == 0) TRACE(EV_EPI_B, i);
  if (!WAIT(&cx.bars->dwbar, i & 1)) return;
  if (tdz < NR) {
    const int rr = tdz >> 6, h = tdz & 63;
    if (rr < Rb && h < p.H) {
      // the four key quarters' partials in a fixed order
      const float s4 = ((dwp[tdz] + dwp[NR + tdz]) + dwp[2 * NR + tdz]) + dwp[3 * NR + tdz];
      const float dwv = s4 * p.sm_scale;
      const long long e = (long long)(row0 + rr) * p.H + h;
      if (p.dw16)
        p.dw16[e] = to_bf16(dwv);
      else
        p.dw[e] = dwv;
    }
  }
  if (tdz == 0) TRACE(EV_EPI_C, i);
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
    const int flags = cx.hdr[ms].flags, c = cx.hdr[ms].c;
    if (flags & F_FIRST) {
      ++i;
      if (!WAIT(&B->qfull[0], i & 1)) return;  // and w
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
      float ad = 0.f;  // dW: this tile's sum of dI relu(z)
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
            ad = fmaf(dA, fmaxf(z0, 0.f), fmaf(dB, fmaxf(z1, 0.f), ad));
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
    // the block's rows, read before the arrive: once the tile's MMAs are
    // complete its record slot may be released and rewritten
    const int row0 = cx.hdr[ms].row0, Rb = cx.hdr[ms].Rb;
    fence_proxy_async_smem();
    mbar_arrive(&B->dzfull);
    if (tdz == 0) TRACE(EV_DZ_DONE, g);
    if (flags & F_LAST) dz_epilogue(p, cx, row0, Rb, c, i, acc0, acc1);
    if (flags & F_END) return;
  }
}

// ------------------------------------------------------------ dK group ----
// dK warp w (0..7): TMEM lane quarter qw = w % 4 (32 columns d), entries
// 64*(w/4) .. +63 of the tile in two chunks of 32.  (Straight from TMEM,
// lane l holds column d of each entry, so each entry's 32 columns could go
// out as one whole-line scalar reduction per warp instruction; built and
// measured, that made the anchor's gemm stage 1106 us against 854: four
// times the reduction instructions per tile held back the dK warps.  The
// transpose through shared memory lets one 16-byte vector reduction per lane
// cover four whole lines.)
__device__ void dk_role(const BParams& p, const Ctx& cx) {
  const int qw = (threadIdx.x >> 5) & 3;
  const int kg = (threadIdx.x - W_DK0 * 32) >> 7;
  float* stage = reinterpret_cast<float*>(cx.smem + OFF_DKST) + ((threadIdx.x >> 5) - W_DK0) * 512;
  Bars* B = cx.bars;
  // the ids' bound: rows of u (deterministic mode) or keys of a batch
  const int idmax = p.u ? (int)(p.dense ? (long long)p.B * p.dense_batch_entries - 1
                                        : p.nblocks * min((long long)p.S_k, (long long)R * p.L) - 1)
                        : p.S_k - 1;
  unsigned nb = 0;  // blocks before this tile's (its parity is what is used)
  for (long long g = 0;; ++g) {
    const int ms = (int)(g % MST);
    if (!WAIT(&B->mfull[ms], (g / MST) & 1)) return;
    const int flags = cx.hdr[ms].flags, c = cx.hdr[ms].c, count = cx.hdr[ms].count, batch = cx.hdr[ms].batch;
    // deterministic: the Q loader's maximum of this block, complete once its
    // q is (the next phase of qfull needs this block's last dK MMA, which
    // needs this role)
    if (p.u && (flags & F_FIRST) && !WAIT(&B->qfull[1], nb & 1)) return;
    const int qe = p.u ? q_exponent(reinterpret_cast<const unsigned*>(cx.smem + OFF_MISC + 8)[nb & 1]) : 0;
    float* base = p.dk + (long long)batch * p.S_k * p.D;
    const int* ids = p.u ? rec_pos(cx, ms) : rec_key(cx, ms);
    if (!WAIT(&B->dkfull, g & 1)) return;
    if (threadIdx.x == W_DK0 * 32) TRACE(EV_DK_FULL, (int)g);
    tc_fence_after();
    const float sc = pow2f(-c) * p.sm_scale;
    // deterministic rows: |dK^T| < 256 * 2^14 * 2^qe (256 products of
    // |dz| < 2^14 and |q| < 2^qe), so 2^-(7+qe) keeps them below 2^15 in
    // fp16; the factor restores the scale (saturated at the largest float,
    // so that a zero row stays zero)
    const float su = pow2f(-7 - qe);
    const float fu = fminf(ldexpf(p.sm_scale, 7 + qe - c), 3.4028235e38f);
    const uint32_t ta = cx.tmem + ((uint32_t)(qw * 32) << 16) + TM_DK;
#pragma unroll 1
    for (int ch = kg * 2; ch < kg * 2 + 2; ++ch) {
      if (ch * 32 >= count) break;  // uniform: the remaining entries are padding
      const int nrow = min(32, count - ch * 32);
      if (p.u)
        dk_chunk_u16(p.u, ids + ch * 32, ta + ch * 32, nrow, su, fu, p.D, qw * 32, stage, idmax, qw == 0);
      else
        dk_chunk_tmem(base, ids + ch * 32, ta + ch * 32, nrow, sc, p.D, qw * 32, stage, idmax);
    }
    tc_fence_before();
    mbar_arrive(&B->dkempty);
    mbar_arrive(&B->mempty[ms]);
    if (threadIdx.x == W_DK0 * 32) TRACE(EV_DK_DONE, (int)g);
    if (flags & F_LAST) ++nb;
    if (flags & F_END) return;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) blk_kernel(const BParams p, const __grid_constant__ CUtensorMap qmap) {
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
    mbar_init(&B->qfull[0], NQT);
    mbar_init(&B->qfull[1], NQT);
    mbar_init(&B->qempty, 1);
    mbar_init(&B->qraw, 1);
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
  const bool run = p.select == nullptr || __ldcg(p.select) == 0u;

  if (!run) {
    // the per-row kernel serves this call
  } else if (warp < W_SCAN) {
    gather_role(p, cx);
  } else if (warp == W_SCAN) {
    scan_role(p, cx);
  } else if (warp == W_MMA) {
    zmma_role(p, cx);  // the whole warp runs the loop; one elected lane issues
  } else if (warp == W_GMMA) {
    gmma_role(p, cx);
  } else if (warp < W_DZ0) {
    q_role(p, cx, &qmap);
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

std::atomic<int> g_attr_pipe[64];

}  // namespace

template <>
cudaError_t launch_blk_pipe<KST, MST>(const blk::BParams& p, const CUtensorMap& qmap, int grid, cudaStream_t st) {
  if (!set_smem_attr((const void*)blk_kernel, SMEM_BYTES, g_attr_pipe)) return cudaErrorInvalidValue;
  return launch_ex(blk_kernel, (unsigned)grid, (unsigned)NTHREADS, SMEM_BYTES, st, true, p, qmap);
}

#if IBWD_PIPE_PRIMARY
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
#endif

}  // namespace ibwd
