// Forward of the lightning indexer on sm_103a: the logits the backward
// differentiates,
//   index_score[t, j] = sum_h w[t,h] relu(q[t,h,:] . k[s,:]),  s = topk_idx[t,j]
// (cudnn-frontend #730 "optimize SM100 gradient kernels", benchmark-harness
// comment: the indexer scores every selected key of a query with one shared
// key head), 0 on padding slots (any id outside [0, S_k)).  Dense variant:
// every key s <= t, scores [B, S, S] with 0 above the diagonal.
//
// The same pipeline as the gemm stage without its backward half: one
// persistent CTA per SM walks its query rows; each row's valid slots are
// compacted into tiles of 128 keys, gathered as bf16 rows by cp.async into a
// 128-byte-swizzled tile, and one tcgen05 MMA per tile computes
// Z^T[128 s, 64 h] = Ksel . Q^T with bf16 operands (q and k as given, no
// conversion) and fp32 accumulation in TMEM.  An epilogue thread per key row
// reduces its Z row against w in registers.
//
// Warp roles (16 warps):
//   0-7   gather: 8 cp.async of 16 B per thread per tile (zero-filled for
//         padding rows and for columns beyond D)
//   8     scan: the row's ids staged by a bulk copy one row ahead, compaction
//         into tile metadata, zeros written for padding slots
//   9     MMA issuer and TMEM owner
//   10-11 Q loader: q[t] by cp.async into the swizzled tile (zero-filled for
//         heads beyond H), w[t] into shared memory
//   12-15 epilogue: Z from TMEM, index_score = sum_h w relu(z)
// Every mbarrier wait is bounded (status bit, abort, drain, TMEM freed).
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace ibwd {
namespace {

constexpr int FKST = 4;  // key-tile stages
constexpr int FMST = 8;  // tile-metadata ring
constexpr int FNTHREADS = 512;
constexpr int FW_GATHER0 = 0, FW_SCAN = 8, FW_MMA = 9, FW_Q0 = 10, FW_EPI0 = 12;
constexpr int FNGT = 256, FNQT = 64, FNET = 128;
constexpr uint32_t FROW_BYTES = 16384;  // one staged id row (topk <= 4096)
constexpr uint32_t FKTILE = kBM * kDP * 2, FKHALF = kBM * 64 * 2;
constexpr uint32_t FQTILE = kHP * kDP * 2, FQHALF = kHP * 64 * 2;

struct FMeta {
  int key[kBM];
  int slot[kBM];
  int r, count, flags;
};
enum { FF_FIRST = 1, FF_LAST = 2, FF_END = 4 };

struct FBars {
  uint64_t kfull[FKST], kempty[FKST];
  uint64_t mfull[FMST], mempty[FMST];
  uint64_t rowfull[2];
  uint64_t qfull[2], qmma[2], qepi[2];
  uint64_t zfull[2], zempty[2];
  uint64_t drain;
};

constexpr uint32_t FOFF_K = 0;
constexpr uint32_t FOFF_Q = FOFF_K + FKST * FKTILE;
constexpr uint32_t FOFF_ROW = FOFF_Q + 2 * FQTILE;
constexpr uint32_t FOFF_META = FOFF_ROW + 2 * FROW_BYTES;
constexpr uint32_t FOFF_W = FOFF_META + FMST * sizeof(FMeta);
constexpr uint32_t FOFF_BARS = FOFF_W + 2 * kHP * 4;
constexpr uint32_t FOFF_MISC = FOFF_BARS + sizeof(FBars);
constexpr uint32_t FSMEM_BYTES = FOFF_MISC + 16 + 1024;  // + alignment slack
static_assert(FOFF_BARS % 8 == 0 && FOFF_ROW % 16 == 0, "alignment");
static_assert(FSMEM_BYTES <= 232448, "shared memory budget");

// kind::f16 instruction descriptor with bf16 A and B, fp32 accumulation.
constexpr uint32_t FID_Z = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(64 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

struct FParams {
  const uint16_t* q;    // bf16 [B, S_q, H, D]
  const uint16_t* k;    // bf16 [B, S_k, D]
  const float* w;       // [B, S_q, H]
  const int32_t* idx;   // [B, S_q, L] or nullptr (dense)
  float* out;           // [B, S_q, L]
  unsigned* status;
  long long rows;
  unsigned long long wait_ns;
  int B, S_q, S_k, H, D, L, dense, staged;
};

struct FCtx {
  uint32_t sbase;
  uint8_t* smem;
  FMeta* meta;
  float* w_s;
  FBars* bars;
  volatile int* abort;
  uint32_t tmem;
  long long nq;
};

#define FWAIT(bar, par) mbar_wait((bar), (par), cx.abort, p.status, p.wait_ns)
#define FWAITW(bar, par) __all_sync(0xffffffffu, FWAIT(bar, par))

__device__ __forceinline__ long long frow(const FCtx& cx, long long i) { return blockIdx.x + i * gridDim.x; }

// ------------------------------------------------------------------ scan --
__device__ void fscan_role(const FParams& p, const FCtx& cx) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  uint8_t* rowbuf = cx.smem + FOFF_ROW;
  long long staged_wait = -1;
  auto issue_row = [&](long long i) {
    if (lane == 0) {
      fence_proxy_async_smem();
      const int buf = (int)(i & 1);
      const uint32_t bytes = (uint32_t)p.L * 4;
      mbar_arrive_expect_tx(&cx.bars->rowfull[buf], bytes);
      bulk_g2s(smem_u32(rowbuf + buf * FROW_BYTES), p.idx + frow(cx, i) * p.L, bytes, &cx.bars->rowfull[buf]);
    }
    staged_wait = i;
  };
  int g = 0;
  if (p.staged && cx.nq > 0) issue_row(0);
  for (long long i = 0; i < cx.nq; ++i) {
    const long long r = frow(cx, i);
    const int t = (int)(r % p.S_q);
    float* orow = p.out + r * p.L;
    const int32_t* ids = nullptr;
    if (!p.dense) {
      if (p.staged) {
        const int buf = (int)(i & 1);
        if (!FWAIT(&cx.bars->rowfull[buf], (uint32_t)((i >> 1) & 1))) goto done;
        staged_wait = -1;
        __syncwarp();
        if (i + 1 < cx.nq) issue_row(i + 1);
        ids = reinterpret_cast<const int32_t*>(rowbuf + buf * FROW_BYTES);
      } else {
        ids = p.idx + r * p.L;
      }
    }
    const int lim = p.dense ? min(p.L, t + 1) : p.L;
    // valid slots of the row, and zeros for its padding slots
    int nv = 0;
    for (int j0 = 0; j0 < p.L; j0 += 32) {
      const int j = j0 + lane;
      bool v = false;
      if (j < lim) v = p.dense ? true : (unsigned)ids[j] < (unsigned)p.S_k;
      if (j < p.L && !v) orow[j] = 0.f;
      nv += __popc(__ballot_sync(0xffffffffu, v));
    }
    const int ntiles = max(1, (nv + kBM - 1) / kBM);
    int jc = 0, skip = 0;
    for (int tt = 0; tt < ntiles; ++tt, ++g) {
      const int ms = g % FMST;
      if (!FWAIT(&cx.bars->mempty[ms], (uint32_t)(((g / FMST) & 1) ^ 1))) goto done;
      FMeta& M = cx.meta[ms];
      int fill = 0;
      while (fill < kBM && jc < lim) {
        const int j = jc + lane;
        int s = 0;
        bool v = false;
        if (j < lim) {
          s = p.dense ? j : ids[j];
          v = p.dense ? true : (unsigned)s < (unsigned)p.S_k;
        }
        const unsigned mask = __ballot_sync(0xffffffffu, v);
        const int tot = __popc(mask), rank = __popc(mask & lt), room = kBM - fill;
        if (v && rank >= skip && rank < skip + room) {
          const int pos = fill + rank - skip;
          M.key[pos] = s;
          M.slot[pos] = j;
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
        M.flags = (tt == 0 ? FF_FIRST : 0) | (tt == ntiles - 1 ? FF_LAST : 0) |
                  ((tt == ntiles - 1 && i == cx.nq - 1) ? FF_END : 0);
      }
      __syncwarp();
      mbar_arrive(&cx.bars->mfull[ms]);
    }
    __syncwarp();
  }
done:
  if (staged_wait >= 0) {
    volatile int never = 0;
    mbar_wait(&cx.bars->rowfull[staged_wait & 1], (uint32_t)((staged_wait >> 1) & 1), &never, p.status, p.wait_ns);
  }
}

// ---------------------------------------------------------------- gather --
// Thread x copies chunk (x % 16) of rows (x / 16) + 16i: every warp
// instruction moves two whole 256-byte key rows into the 128-byte-swizzle
// layout (half chunk / 8, XOR (chunk % 8) ^ (row % 8)).
__device__ void fgather_role(const FParams& p, const FCtx& cx) {
  const int x = threadIdx.x - FW_GATHER0 * 32;  // 0..255
  const int rsub = x >> 4, ch = x & 15;         // rsub 0..15
  const uint32_t dst_off = (ch >> 3) * FKHALF + rsub * 128 + (((ch & 7) ^ (rsub & 7)) << 4);
  const uint32_t cbytes = ch * 8 < p.D ? 16u : 0u;  // columns beyond D are zero-filled
  for (int g = 0;; ++g) {
    const int ms = g % FMST;
    if (!FWAIT(&cx.bars->mfull[ms], (uint32_t)((g / FMST) & 1))) break;
    const FMeta& M = cx.meta[ms];
    const int count = M.count, flags = M.flags;
    const long long b = M.r / p.S_q;
    const int st = g % FKST;
    if (!FWAIT(&cx.bars->kempty[st], (uint32_t)(((g / FKST) & 1) ^ 1))) break;
    const uint32_t kbase = cx.sbase + FOFF_K + st * FKTILE + dst_off;
    const uint16_t* kb = p.k + b * p.S_k * p.D + ch * 8;
#pragma unroll
    for (int i = 0; i < kBM / 16; ++i) {
      const int row = rsub + 16 * i;
      const bool live = row < count;
      // padding rows are zero-filled (no bytes read from the valid base address)
      cp_async16(kbase + i * 2048, live ? kb + (long long)M.key[row] * p.D : p.k, live ? cbytes : 0u);
    }
    cp_async_mbar_arrive_noinc(&cx.bars->kfull[st]);
    if (flags & FF_END) break;
  }
  cp_async_wait_all();
}

// -------------------------------------------------------------- Q loader --
__device__ void fq_role(const FParams& p, const FCtx& cx) {
  const int tid = threadIdx.x - FW_Q0 * 32;  // 0..63
  for (long long i = 0; i < cx.nq; ++i) {
    const int qb = (int)(i & 1);
    // the buffer's previous row (i - 2): its MMAs and its epilogue are done
    if (i >= 2 && (!FWAIT(&cx.bars->qmma[qb], (uint32_t)(((i - 2) >> 1) & 1)) ||
                   !FWAIT(&cx.bars->qepi[qb], (uint32_t)(((i - 2) >> 1) & 1))))
      return;
    const long long r = frow(cx, i);
    const uint16_t* qr = p.q + r * p.H * p.D;
    const uint32_t qs = cx.sbase + FOFF_Q + qb * FQTILE;
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int x = tid + it * FNQT;  // 16-byte chunk: head h, column chunk ch
      const int h = x >> 4, ch = x & 15;
      const bool live = h < p.H && ch * 8 < p.D;
      const uint32_t dst = qs + (ch >> 3) * FQHALF + h * 128 + (((ch & 7) ^ (h & 7)) << 4);
      cp_async16(dst, live ? qr + h * p.D + ch * 8 : p.q, live ? 16u : 0u);
    }
    cp_async_mbar_arrive_noinc(&cx.bars->qfull[qb]);
    cx.w_s[qb * kHP + tid] = tid < p.H ? __ldg(p.w + r * p.H + tid) : 0.f;
    mbar_arrive(&cx.bars->qfull[qb]);
  }
  cp_async_wait_all();
}

// ------------------------------------------------------------------- MMA --
__device__ void fmma_role(const FParams& p, const FCtx& cx) {
  FBars* B = cx.bars;
  long long iq = -1;
  for (int g = 0;; ++g) {
    if (!FWAITW(&B->mfull[g % FMST], (uint32_t)((g / FMST) & 1))) break;
    const int flags = cx.meta[g % FMST].flags;
    if (flags & FF_FIRST) {
      ++iq;
      if (!FWAITW(&B->qfull[iq & 1], (uint32_t)((iq >> 1) & 1))) break;
    }
    if (!FWAITW(&B->kfull[g % FKST], (uint32_t)((g / FKST) & 1))) break;
    if (g >= 2 && !FWAITW(&B->zempty[g & 1], (uint32_t)(((g >> 1) & 1) ^ 1))) break;
    // the tiles were written by cp.async (generic proxy): order them before
    // the tensor core's reads
    fence_proxy_async_smem();
    tc_fence_after();
    const uint64_t a0 = sw128_desc(cx.sbase + FOFF_K + (g % FKST) * FKTILE, 16, 1024);
    const uint64_t b0 = sw128_desc(cx.sbase + FOFF_Q + (int)(iq & 1) * FQTILE, 16, 1024);
    const uint32_t d = cx.tmem + (uint32_t)(g & 1) * 64;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)  // K = D = 128 in steps of 16
      umma_f16_elect(d, a0 + (((kk >> 2) * FKHALF + (kk & 3) * 32) >> 4),
                     b0 + (((kk >> 2) * FQHALF + (kk & 3) * 32) >> 4), FID_Z, kk > 0);
    umma_commit_elect(&B->zfull[g & 1]);
    umma_commit_elect(&B->kempty[g % FKST]);
    if (flags & FF_LAST) umma_commit_elect(&B->qmma[iq & 1]);
    if (flags & FF_END) break;
  }
  // every MMA issued so far completes before TMEM can be released
  __syncwarp();
  umma_commit_elect(&B->drain);
  volatile int never = 0;
  mbar_wait(&B->drain, 0, &never, p.status, p.wait_ns);
}

// -------------------------------------------------------------- epilogue --
__device__ void fepi_role(const FParams& p, const FCtx& cx) {
  const int qw = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int s = qw * 32 + lane;  // tile row = TMEM lane
  long long iq = -1;
  for (int g = 0;; ++g) {
    const int ms = g % FMST;
    if (!FWAIT(&cx.bars->mfull[ms], (uint32_t)((g / FMST) & 1))) return;
    const FMeta& M = cx.meta[ms];
    const int flags = M.flags, count = M.count;
    const long long r = M.r;
    const int slot = s < count ? M.slot[s] : 0;
    if (flags & FF_FIRST) {
      ++iq;
      if (!FWAIT(&cx.bars->qfull[iq & 1], (uint32_t)((iq >> 1) & 1))) return;  // w of the row
    }
    if (!FWAIT(&cx.bars->zfull[g & 1], (uint32_t)((g >> 1) & 1))) return;
    tc_fence_after();
    const uint32_t za = cx.tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(g & 1) * 64;
    float z0[32], z1[32];
    tmem_ld32(za, z0);
    tmem_ld32(za + 32, z1);
    tmem_wait_ld_dep(z0);
    tmem_wait_ld_dep(z1);
    tc_fence_before();
    mbar_arrive(&cx.bars->zempty[g & 1]);
    const float* wr = cx.w_s + (iq & 1) * kHP;
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < 32; ++h) acc = fmaf(wr[h], fmaxf(z0[h], 0.f), acc);
#pragma unroll
    for (int h = 0; h < 32; ++h) acc = fmaf(wr[32 + h], fmaxf(z1[h], 0.f), acc);
    if (s < count) p.out[r * p.L + slot] = acc;
    if (flags & FF_LAST) mbar_arrive(&cx.bars->qepi[iq & 1]);
    mbar_arrive(&cx.bars->mempty[ms]);
    if (flags & FF_END) return;
  }
}

__global__ void __launch_bounds__(FNTHREADS, 1) fwd_kernel(const FParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FCtx cx;
  cx.smem = smem;
  cx.sbase = smem_u32(smem);
  cx.meta = reinterpret_cast<FMeta*>(smem + FOFF_META);
  cx.w_s = reinterpret_cast<float*>(smem + FOFF_W);
  cx.bars = reinterpret_cast<FBars*>(smem + FOFF_BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + FOFF_MISC);
  cx.abort = reinterpret_cast<volatile int*>(smem + FOFF_MISC + 4);
  cx.nq = (p.rows - (long long)blockIdx.x + gridDim.x - 1) / gridDim.x;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    FBars* B = cx.bars;
    for (int i = 0; i < FKST; ++i) {
      mbar_init(&B->kfull[i], FNGT);
      mbar_init(&B->kempty[i], 1);
    }
    for (int i = 0; i < FMST; ++i) {
      mbar_init(&B->mfull[i], 32);
      mbar_init(&B->mempty[i], FNET);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->rowfull[i], 1);
      mbar_init(&B->qfull[i], 2 * FNQT);  // each Q thread: its copies landed, then its w store
      mbar_init(&B->qmma[i], 1);
      mbar_init(&B->qepi[i], FNET);
      mbar_init(&B->zfull[i], 1);
      mbar_init(&B->zempty[i], FNET);
    }
    mbar_init(&B->drain, 1);
    *cx.abort = 0;
    fence_barrier_init();
  }
  if (warp == FW_MMA) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  if (cx.nq > 0) {
    if (warp < FW_SCAN)
      fgather_role(p, cx);
    else if (warp == FW_SCAN)
      fscan_role(p, cx);
    else if (warp == FW_MMA)
      fmma_role(p, cx);
    else if (warp < FW_EPI0)
      fq_role(p, cx);
    else
      fepi_role(p, cx);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == FW_MMA) tmem_dealloc(cx.tmem, 128);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t st) {
  static std::atomic<bool> attr_set[64];  // per device; setting the attribute twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FSMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  FParams p{};
  p.q = a.q;
  p.k = a.k;
  p.w = a.w;
  p.idx = a.idx;
  p.out = a.out;
  p.status = a.status;
  p.rows = (long long)a.B * a.S_q;
  p.wait_ns = 2000000000ull;
  p.B = a.B;
  p.S_q = a.S_q;
  p.S_k = a.S_k;
  p.H = a.H;
  p.D = a.D;
  p.L = a.L;
  p.dense = a.idx == nullptr;
  p.staged = !p.dense && (size_t)a.L * 4 <= FROW_BYTES && a.L % 4 == 0 && (uintptr_t)a.idx % 16 == 0;
  const int grid = (int)std::min<long long>(a.num_sms, p.rows);
  fwd_kernel<<<grid, FNTHREADS, FSMEM_BYTES, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ibwd
