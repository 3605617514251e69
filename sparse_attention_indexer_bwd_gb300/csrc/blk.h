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
#pragma once
#include <atomic>

#include <cuda.h>  // CUtensorMap

#include "kcommon.cuh"

namespace ibwd {
namespace blk {

constexpr int R = kBlkRows;   // query rows per block
constexpr int NR = R * kHP;   // (r,h) rows of a block: 256
constexpr unsigned FULL = 0xffffffffu;
// A tile record: int key[128] | float dis[R][128] | int pos[128] (the last
// only in deterministic mode): byte offsets, and the size of a whole record
constexpr int REC_KEY = 0, REC_DIS = 512, REC_POS = 2560;
constexpr uint32_t REC_BYTES = 3072;

// A block's q rows as the gemm kernel's Q operand: fp16, [d-half][(r,h) =
// 64r + h][128 B], each 128-byte row's 16-byte chunks in the 128-byte swizzle
// (chunk c of row n at (c ^ n % 8) * 16); rows past the block, heads past H
// and columns past D zero.  Two TMA tile loads of q (bf16) land in exactly
// this layout; the kernel converts them to fp16 in place.
constexpr uint32_t QIMG_HALF = NR * 128;  // one 64-column half: 32 KB
constexpr uint32_t QIMG_BYTES = 2 * QIMG_HALF;

struct BParams {
  const uint16_t* q;   // bf16 [rows, H, D]
  const __half* k16;   // [B][S_k + 1][128]; row S_k of each batch is zero
  const float* w;      // [rows, H]
  const float* dI;     // dense: [rows, S] (sparse blocks read their tile records instead)
  const char* rec;     // sparse: tile records
  const int4* binfo;   // per block {tiles, c, entries, 0}
  const int* border;   // sparse: processing order of the blocks
  float* dq;
  float* dw;
  float* dk;           // [B, S_k, D] (atomic mode)
  char* u;             // deterministic: per-entry dK rows in key order (u_row_bytes(D) each), or nullptr
  uint16_t* dq16;      // bf16 outputs instead of dq / dw when set
  uint16_t* dw16;
  unsigned* sched;     // block counter, zeroed by the k conversion kernel
  unsigned* status;
  long long nblocks;
  unsigned long long wait_ns;   // limit of the roles' waits
  unsigned long long drain_ns;  // limit of the drains of issued copies and MMAs before exit
  float sm_scale;               // logit scale s > 0: every output is s times the unscaled one
  int test_stall;               // test of the timeout path: the record producer publishes nothing
  const unsigned* select;       // if set: the kernel runs only when *select == 0 (1 selects the per-row kernel)
  int B, S_q, S_k, H, D, L;
  int dense, nbpb, tcap, rstride;
  long long dense_batch_entries;  // deterministic dense: entries (rows of u) per batch
};

// Raises a kernel's dynamic shared-memory limit once per device (raising it
// twice is harmless).
inline bool set_smem_attr(const void* fn, size_t bytes, std::atomic<int>* done) {
  // per device; raising the attribute twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
  if (done[dev].load(std::memory_order_acquire) >= (int)bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) return false;
  done[dev].store((int)bytes, std::memory_order_release);
  return true;
}

}  // namespace blk

// The gemm kernel for one pair of pipeline depths: KST K-tile stages and MST
// tile-record slots.  <2, 4> is the one the library runs (blk_pipe.cu);
// <1, 2> (blk_pipe_shallow.cu) exists to test that the results do not depend
// on the depths.
// qmap: q as a 4-d bf16 tensor [B][S_q][H][D] with boxes of 4 rows x 64
// heads x 64 columns and the 128-byte swizzle (one block's Q operand half).
template <int KST, int MST>
cudaError_t launch_blk_pipe(const blk::BParams& p, const CUtensorMap& qmap, int grid, cudaStream_t st);
template <>
cudaError_t launch_blk_pipe<2, 4>(const blk::BParams& p, const CUtensorMap& qmap, int grid, cudaStream_t st);
template <>
cudaError_t launch_blk_pipe<1, 2>(const blk::BParams& p, const CUtensorMap& qmap, int grid, cudaStream_t st);

}  // namespace ibwd
