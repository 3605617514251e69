// Score-grad of the lightning-indexer backward (kernel 1).
//
// cudnn-frontend #730 "optimize SM100 gradient kernels" (walkthrough): kernel 1
// turns the forward indexer logits (index_score, read only) and the target
// distribution (attn_score) into the gradient signal dI, written in place over
// attn_score; the same change fuses the zeroing of the fp32 dK accumulator
// into this launch.  #549 names the kernel kernel_score_grad.  The pages give
// no formula; the plain reading is the gradient of the row-mean KL divergence
// KL(ahat || softmax(I)):
//   p_j    = exp(I_j - m) / sum_valid exp(I - m)      (m = max over valid j)
//   ahat_j = a_j / sum_valid a                        (0 when the sum is 0)
//   dI_j   = grad_scale * (p_j - ahat_j) / S_q         (0 on padding slots)
// A slot is valid iff its id lies in [0, S_k) (dense rows: iff j <= t); with
// global ids, a row of batch b subtracts b*S_k from each id first.
// Padding slots are selected out, never multiplied by a mask, so NaN or
// garbage there never reaches dI.
//
// HBM-bound: 16 bytes per slot (read I, a, id; write dI).  Sparse rows of
// 128..2048 slots go to a persistent kernel that streams rows through a
// three-deep shared-memory ring of bulk copies; other shapes use a group of
// 32*W threads per row that keeps the row in registers (NV float4 per thread
// per array).  All reductions are fixed-order (bitwise reproducible).
#include <algorithm>
#include <atomic>

#include "internal.h"

namespace ibwd {
namespace {

constexpr int BLOCK = 256;

// Lets the kernel queued after this one, when it is launched with
// programmatic stream serialization, start launching now; it still waits for
// this grid to complete before it reads anything this grid writes.
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

template <int W>
struct RowReduce {
  // Sum/max over the row group (W warps) in a fixed order.
  __device__ static float sum(float v, float* sh, int wig) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (W == 1) return v;
    const int lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) sh[wig] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) t += sh[i];
    return t;
  }
  __device__ static float max(float v, float* sh, int wig) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (W == 1) return v;
    const int lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) sh[wig] = v;
    __syncthreads();
    float t = -INFINITY;
#pragma unroll
    for (int i = 0; i < W; ++i) t = fmaxf(t, sh[i]);
    return t;
  }
};

// NV float4 per thread per array; W warps per row; BLOCK/(32W) rows per block.
template <int NV, int W>
__global__ void __launch_bounds__(BLOCK) score_grad_vec(ScoreGradArgs a, long long row_blocks) {
  allow_dependent_launch();
  __shared__ float red[BLOCK / 32];
  constexpr int G = 32 * W;                 // threads per row
  constexpr int RPB = BLOCK / G;            // rows per block
  if ((long long)blockIdx.x >= row_blocks) {
    // trailing blocks zero the dK accumulator
    if (a.dk_zero) {
      const long long nb = gridDim.x - row_blocks;
      const long long n4 = a.dk_numel / 4;
      float4* d4 = reinterpret_cast<float4*>(a.dk_zero);
      for (long long x = (blockIdx.x - row_blocks) * (long long)BLOCK + threadIdx.x; x < n4; x += nb * BLOCK)
        d4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (long long x = n4 * 4 + (blockIdx.x - row_blocks) * (long long)BLOCK + threadIdx.x; x < a.dk_numel;
           x += nb * BLOCK)
        a.dk_zero[x] = 0.f;
    }
    return;
  }
  const int grp = threadIdx.x / G;          // row within the block
  const int gt = threadIdx.x % G;           // thread within the row group
  const int wig = gt / 32;                  // warp within the row group
  float* sh = red + grp * W;
  const long long r = (long long)blockIdx.x * RPB + grp;
  const bool live = r < a.rows;             // uniform per row group
  const long long rr = live ? r : 0;
  const int L4 = a.L / 4;
  const float4* I4 = reinterpret_cast<const float4*>(a.index_score + rr * a.L);
  float4* A4 = reinterpret_cast<float4*>(a.attn_score + rr * a.L);
  const int4* X4 = a.idx ? reinterpret_cast<const int4*>(a.idx + rr * a.L) : nullptr;
  const int t = (int)(rr % a.S_q);
  const int lim = a.idx ? a.L : min(a.L, t + 1);  // dense: slots beyond t are padding
  const int off = a.ids_global ? ((int)rr / a.S_q) * a.S_k : 0;  // rows < 2^31

  float iv[NV][4], av[NV][4];
  bool vv[NV][4];
  float m = -INFINITY, sa = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v4 = gt + k * G;
    const bool in = live && v4 < L4 && v4 * 4 < lim;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
    int4 id = make_int4(-1, -1, -1, -1);
    if (in) {
      x = __ldcs(I4 + v4);
      y = __ldcs(A4 + v4);
      if (X4) id = __ldcs(X4 + v4);
    }
    const float xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
    const int ids[4] = {id.x, id.y, id.z, id.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = v4 * 4 + e;
      const bool v = in && (X4 ? ((unsigned)ids[e] - (unsigned)off < (unsigned)a.S_k) : (j < lim));
      vv[k][e] = v;
      iv[k][e] = xs[e];
      av[k][e] = ys[e];
      if (v) {
        m = fmaxf(m, xs[e]);
        sa += ys[e];
      }
    }
  }
  m = RowReduce<W>::max(m, sh, wig);
  sa = RowReduce<W>::sum(sa, sh, wig);
  float z = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float ex = vv[k][e] ? expf(iv[k][e] - m) : 0.f;
      iv[k][e] = ex;
      z += ex;
    }
  z = RowReduce<W>::sum(z, sh, wig);
  if (!live) return;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v4 = gt + k * G;
    if (v4 >= L4) continue;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float ahat = sa != 0.f ? __fdiv_rn(av[k][e], sa) : 0.f;
      o[e] = vv[k][e] ? a.scale * (__fdiv_rn(iv[k][e], z) - ahat) : 0.f;
    }
    __stcs(A4 + v4, make_float4(o[0], o[1], o[2], o[3]));
  }
}

// Any row length: one block per row, three strided passes.
__global__ void __launch_bounds__(BLOCK) score_grad_generic(ScoreGradArgs a, long long row_blocks) {
  allow_dependent_launch();
  __shared__ float red[BLOCK / 32];
  if ((long long)blockIdx.x >= row_blocks) {
    if (a.dk_zero) {
      const long long nb = gridDim.x - row_blocks;
      for (long long x = (blockIdx.x - row_blocks) * (long long)BLOCK + threadIdx.x; x < a.dk_numel; x += nb * BLOCK)
        a.dk_zero[x] = 0.f;
    }
    return;
  }
  const long long r = blockIdx.x;
  const float* I = a.index_score + r * a.L;
  float* A = a.attn_score + r * a.L;
  const int32_t* X = a.idx ? a.idx + r * a.L : nullptr;
  const int t = (int)(r % a.S_q);
  const int lim = a.idx ? a.L : min(a.L, t + 1);
  const int off = a.ids_global ? ((int)r / a.S_q) * a.S_k : 0;  // rows < 2^31
  auto valid = [&](int j) { return X ? ((unsigned)X[j] - (unsigned)off < (unsigned)a.S_k) : (j < lim); };
  auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float u = __shfl_xor_sync(0xffffffffu, v, o);
      v = is_max ? fmaxf(v, u) : v + u;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t2 = is_max ? -INFINITY : 0.f;
    for (int i = 0; i < BLOCK / 32; ++i) t2 = is_max ? fmaxf(t2, red[i]) : t2 + red[i];
    return t2;
  };
  float m = -INFINITY, sa = 0.f;
  for (int j = threadIdx.x; j < a.L; j += BLOCK)
    if (valid(j)) {
      m = fmaxf(m, I[j]);
      sa += A[j];
    }
  m = block_reduce(m, true);
  sa = block_reduce(sa, false);
  float z = 0.f;
  for (int j = threadIdx.x; j < a.L; j += BLOCK)
    if (valid(j)) z += expf(I[j] - m);
  z = block_reduce(z, false);
  for (int j = threadIdx.x; j < a.L; j += BLOCK) {
    float o = 0.f;
    if (valid(j)) {
      const float ahat = sa != 0.f ? __fdiv_rn(A[j], sa) : 0.f;
      o = a.scale * (__fdiv_rn(expf(I[j] - m), z) - ahat);
    }
    A[j] = o;
  }
}

// ------------------------------------------------------- staged rows ---
// Persistent variant: a CTA of L/4 threads owns one row at a time, one float4
// of each array per thread.  Thread 0 keeps up to NSTG rows in flight in
// shared memory (bulk copies of the row's index_score, attn_score and, for
// sparse rows, ids: 12 bytes per slot; dense rows copy only their causal
// prefix of the two score arrays), so HBM streams while the block reduces;
// dI goes out with 16-byte streaming stores (zeros above a dense row's
// diagonal).
constexpr int NSTG = 3;

__device__ __forceinline__ uint32_t sg_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void sg_bulk(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(sg_smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool sg_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sg_smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
// bounded (2 s of %globaltimer) wait for a stage
__device__ __forceinline__ bool sg_wait(uint64_t* bar, uint32_t parity) {
  if (sg_try(bar, parity)) return true;
  uint64_t t0, t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    if (sg_try(bar, parity)) return true;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (t1 - t0 > 2000000000ull) return false;
  }
}

// NV float4 of each array per thread: L = 4 * NV * blockDim.x.  GLOBAL: the
// ids are global (a.ids_global), kept out of the other instances.
template <int NV, bool GLOBAL>
__global__ void __launch_bounds__(512, NV == 1 ? 3 : 2) score_grad_staged(ScoreGradArgs a) {
  allow_dependent_launch();
  extern __shared__ __align__(16) uint8_t sg_smem[];
  __shared__ uint64_t full[NSTG];
  __shared__ float red[32], red2[32];
  const int L = a.L, L4 = L / 4;
  const bool dense = a.idx == nullptr;
  (void)L4;
  const uint32_t row_bytes = (uint32_t)L * 4;
  const uint32_t stage_bytes = (dense ? 2 : 3) * row_bytes;  // I | attn [| ids]
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  // zero this CTA's share of dK first
  if (a.dk_zero) {
    const long long n4 = a.dk_numel / 4;
    float4* d4 = reinterpret_cast<float4*>(a.dk_zero);
    for (long long x = (long long)blockIdx.x * blockDim.x + tid; x < n4; x += (long long)gridDim.x * blockDim.x)
      d4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long x = n4 * 4 + (long long)blockIdx.x * blockDim.x + tid; x < a.dk_numel;
         x += (long long)gridDim.x * blockDim.x)
      a.dk_zero[x] = 0.f;
  }
  if (tid == 0) {
    for (int s = 0; s < NSTG; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sg_smem_u32(&full[s])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const long long G = gridDim.x;
  auto issue = [&](long long i) {  // row blockIdx.x + i*G into stage i % NSTG (thread 0)
    const long long r = blockIdx.x + i * G;
    const int s = (int)(i % NSTG);
    const uint32_t dst = sg_smem_u32(sg_smem + s * stage_bytes);
    // dense rows: only slots 0..t hold scores (rounded up to 16 bytes)
    const uint32_t bytes =
        dense ? (uint32_t)(((min(L, (int)(r % a.S_q) + 1) * 4) + 15) & ~15) : row_bytes;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sg_smem_u32(&full[s])),
                 "r"((dense ? 2 : 3) * bytes)
                 : "memory");
    sg_bulk(dst, a.index_score + r * L, bytes, &full[s]);
    sg_bulk(dst + row_bytes, a.attn_score + r * L, bytes, &full[s]);
    if (!dense) sg_bulk(dst + 2 * row_bytes, a.idx + r * L, bytes, &full[s]);
  };
  const long long nrows = (a.rows - blockIdx.x + G - 1) / G;
  if (tid == 0)
    for (long long i = 0; i < nrows && i < NSTG; ++i) issue(i);
  long long issued = nrows < NSTG ? nrows : NSTG;
  auto block_sum = [&](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = 0.f;
    for (int k = 0; k < nw; ++k) t += red[k];
    __syncthreads();
    return t;
  };
  // max of m and sum of s over the block, in one exchange
  auto block_max_sum = [&](float& m, float& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
    }
    if (lane == 0) {
      red[wid] = m;
      red2[wid] = sm;
    }
    __syncthreads();
    float tm = -INFINITY, ts = 0.f;
    for (int k = 0; k < nw; ++k) {
      tm = fmaxf(tm, red[k]);
      ts += red2[k];
    }
    __syncthreads();
    m = tm;
    sm = ts;
  };
  bool aborted = false;
  for (long long i = 0; i < nrows; ++i) {
    const int s = (int)(i % NSTG);
    const bool ok = sg_wait(&full[s], (uint32_t)((i / NSTG) & 1));
    if (!__syncthreads_and(ok)) {
      aborted = true;
      break;
    }
    const long long r = blockIdx.x + i * G;
    const uint8_t* st = sg_smem + s * stage_bytes;
    const int lim = dense ? min(L, (int)(r % a.S_q) + 1) : L;  // dense: slots beyond t are padding
    const int off = GLOBAL ? ((int)r / a.S_q) * a.S_k : 0;  // rows < 2^31
    float xs[NV][4], ys[NV][4];
    int ids[NV][4];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v4 = tid + k * (int)blockDim.x;  // this thread's k-th float4 of the row
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
      int4 id = make_int4(-1, -1, -1, -1);
      if (v4 < L4 && v4 * 4 < lim) {
        x = reinterpret_cast<const float4*>(st)[v4];
        y = reinterpret_cast<const float4*>(st + row_bytes)[v4];
        if (!dense) id = reinterpret_cast<const int4*>(st + 2 * row_bytes)[v4];
      }
      xs[k][0] = x.x; xs[k][1] = x.y; xs[k][2] = x.z; xs[k][3] = x.w;
      ys[k][0] = y.x; ys[k][1] = y.y; ys[k][2] = y.z; ys[k][3] = y.w;
      ids[k][0] = id.x; ids[k][1] = id.y; ids[k][2] = id.z; ids[k][3] = id.w;
    }
    __syncthreads();  // the stage is free: refill it with row i + NSTG
    if (tid == 0 && issued < nrows) {
      // the block's generic reads of the stage precede the async-proxy writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(issued);
      ++issued;
    }
    bool vv[NV][4];
    float m = -INFINITY, sa = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v4 = tid + k * (int)blockDim.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        vv[k][e] = v4 < L4 && (dense ? v4 * 4 + e < lim : (unsigned)ids[k][e] - (unsigned)off < (unsigned)a.S_k);
        if (vv[k][e]) {
          m = fmaxf(m, xs[k][e]);
          sa += ys[k][e];
        }
      }
    }
    block_max_sum(m, sa);
    float z = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xs[k][e] = vv[k][e] ? expf(xs[k][e] - m) : 0.f;  // now exp(x - max)
        z += xs[k][e];
      }
    z = block_sum(z);
    // one reciprocal per row (the quotients differ from IEEE division by at
    // most one rounding)
    const float rz = 1.0f / z, ra = sa != 0.f ? 1.0f / sa : 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v4 = tid + k * (int)blockDim.x;
      if (v4 < L4) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = vv[k][e] ? a.scale * (xs[k][e] * rz - ys[k][e] * ra) : 0.f;
        __stcs(reinterpret_cast<float4*>(a.attn_score + r * L) + v4, make_float4(o[0], o[1], o[2], o[3]));
      }
    }
  }
  if (aborted) {
    if (tid == 0) atomicOr(a.status, 1u);
    // copies still in flight land before the CTA exits (bounded)
    __syncthreads();
    if (tid == 0)
      for (long long i = 0; i < issued; ++i) (void)sg_wait(&full[i % NSTG], (uint32_t)((i / NSTG) & 1));
  }
}

template <int NV, int W>
cudaError_t launch_vec(const ScoreGradArgs& a, int zero_blocks, cudaStream_t st) {
  constexpr int RPB = BLOCK / (32 * W);
  const long long row_blocks = (a.rows + RPB - 1) / RPB;
  score_grad_vec<NV, W><<<(unsigned)(row_blocks + zero_blocks), BLOCK, 0, st>>>(a, row_blocks);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_grad(const ScoreGradArgs& a, cudaStream_t st) {
  const int zero_blocks = a.dk_zero ? (int)std::min<long long>(256, (a.dk_numel / 4 + BLOCK - 1) / BLOCK + 1) : 0;
  const bool aligned = (a.L % 4 == 0) && ((uintptr_t)a.index_score % 16 == 0) &&
                       ((uintptr_t)a.attn_score % 16 == 0) && (!a.idx || (uintptr_t)a.idx % 16 == 0) &&
                       (!a.dk_zero || (uintptr_t)a.dk_zero % 16 == 0);
  // rows of 256..2048 slots (sparse) or 256..4096 (dense), a multiple of 128:
  // the staged kernel (one float4 per thread per array; two beyond 2048
  // slots).  Shorter rows are packed eight to a CTA, one warp each, in
  // registers (vec<1, 1>: 19 against 22 us for the staged kernel's one-warp
  // CTAs at uniform top-128)
  const int lmax = a.idx ? 2048 : 4096;
  const int nv = a.L > 2048 ? 2 : 1;
  if (aligned && a.L % (128 * nv) == 0 && a.L >= 256 && a.L <= lmax && a.status && a.num_sms > 0) {
    const int threads = a.L / (4 * nv);
    const size_t smem = (size_t)NSTG * (a.idx ? 12 : 8) * a.L;
    static std::atomic<bool> attr_done[64];  // per device; setting the attribute twice is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(score_grad_staged<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           NSTG * 12 * 2048);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(score_grad_staged<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               NSTG * 12 * 2048);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(score_grad_staged<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               NSTG * 8 * 4096);
      if (e != cudaSuccess) return e;
      attr_done[dev].store(true, std::memory_order_release);
    }
    // sparse rows take NV = 1 (L <= 2048); global ids only exist for them
    void (*kern)(ScoreGradArgs) = nv == 2 ? score_grad_staged<2, false>
                                  : (a.idx && a.ids_global) ? score_grad_staged<1, true>
                                                            : score_grad_staged<1, false>;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long long grid = std::min<long long>(a.rows, (long long)a.num_sms * per_sm);
    kern<<<(unsigned)grid, threads, smem, st>>>(a);
    return cudaGetLastError();
  }
  if (aligned) {
    const int L = a.L;
    if (L <= 128) return launch_vec<1, 1>(a, zero_blocks, st);
    if (L <= 256) return launch_vec<2, 1>(a, zero_blocks, st);
    if (L <= 512) return launch_vec<4, 1>(a, zero_blocks, st);
    if (L <= 1024) return launch_vec<8, 1>(a, zero_blocks, st);
    if (L <= 2048) return launch_vec<8, 2>(a, zero_blocks, st);
    if (L <= 4096) return launch_vec<8, 4>(a, zero_blocks, st);
    if (L <= 8192) return launch_vec<8, 8>(a, zero_blocks, st);
  }
  score_grad_generic<<<(unsigned)(a.rows + zero_blocks), BLOCK, 0, st>>>(a, a.rows);
  return cudaGetLastError();
}

}  // namespace ibwd
