// Launchers shared between the translation units of libindexer_bwd.so.
// Each returns a cudaError_t from the launch (cudaSuccess when queued).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace ibwd {

// Padded tile geometry of the gemm-stage kernel.
constexpr int kBM = 128;  // keys per tile (an MMA dimension of Z and dK)
constexpr int kDP = 128;  // head dim padded to 128 (the MMA M dimension for dQ and dK)
constexpr int kHP = 64;   // indexer heads padded to 64
constexpr int kBlkRows = 4;     // query rows per block of the gemm stage
constexpr int kSortBlocks = 2;  // blocks per chunk of the deterministic mode's key sort
// Bytes of one deterministic-mode dK row: D fp16 values padded to whole
// 32-byte sectors, then one sector whose first word is the row's fp32
// restoring factor (the rest zero).  The gemm kernel writes every byte of a
// row at once, so no sector is left partly written.
__host__ __device__ constexpr int u_row_bytes(int D) { return ((2 * D + 31) & ~31) + 32; }
// The per-call counter block (256 bytes at the start of the gemm stage's
// workspace): words the k conversion kernel zeroes, and the deterministic
// sort's CTA counter among them.
constexpr int kSchedWords = 11;
constexpr int kSchedDetScan = 10;

struct ScoreGradArgs {
  const float* index_score;  // [rows, L]
  float* attn_score;         // [rows, L], overwritten with dI
  const int32_t* idx;        // [rows, L] or nullptr for the dense variant
  long long rows;            // B * S_q
  int L;                     // slots per row: topk (sparse) or S (dense)
  int S_q, S_k;
  float scale;               // grad_scale / S_q
  float* dk_zero;            // optional buffer zeroed by the same launch
  long long dk_numel;
  unsigned* status;          // device status word (a bounded wait that gave up)
  int num_sms;
  int ids_global;            // ids index the flattened [B*S_k] keys: slot id of a row of batch b
                             // is key id - b*S_k, valid iff that lies in [0, S_k)
};
cudaError_t launch_score_grad(const ScoreGradArgs& a, cudaStream_t st);

struct GemmArgs {
  const uint16_t* q;     // bf16 [rows, H, D]
  const uint16_t* k;     // bf16 [B, S_k, D]
  const float* w;        // [rows, H]
  const float* dI;       // [rows, L]
  const int32_t* idx;    // [rows, L] or nullptr (dense: key j of row t is valid iff j <= t)
  float* dq;             // [rows, H, D]
  float* dw;             // [rows, H]
  float* dk;             // [B, S_k, D]: accumulated (atomic) or overwritten (deterministic)
  int B, S_q, S_k, H, D, L;
  int deterministic;
  void* ws;              // workspace (layout from gemm_workspace_layout)
  size_t ws_bytes;
  unsigned* status;      // device status word
  int num_sms;
  int after_score_grad;  // queued right after this library's score-grad kernel (same stream)
  int ids_global;        // as in ScoreGradArgs
  uint16_t* dq16;        // if set: dq written here as bf16 (round to nearest even) instead of to dq
  uint16_t* dw16;        // if set: dw likewise
  uint16_t* dk16;        // if set: bf16 copy of the final dk, written after it
  float sm_scale;        // logit scale s (> 0; 0 reads as 1): dq, dw, dk are s times the unscaled results
  cudaStream_t side;     // a second stream of the device
  cudaEvent_t ev_fork;
  // set by the one-call entry points, which fork the side stream before
  // their score-grad (ev_fork): the k copy and the kernel choice then run on
  // it beside the score-grad, and ev_sel (recorded after the choice) holds
  // back the union pass until the choice is made
  int early_side;
  cudaEvent_t ev_sel;
};

// Workspace of the gemm stage (indexer_bwd_gemm and the one-call forms).
// The query rows are taken in blocks of kBlkRows consecutive rows of one
// batch; a sparse block's work list is the union of its rows' valid keys,
// stored as tile records of 128 entries:
//   int key[128] | float dis[kBlkRows][128] | int pos[128] (deterministic)
// (dis[r][e]: the sum of dI over row r's slots selecting key e, 0 when row r
// does not select it; padding entries have key S_k and dis 0; pos[e]: the
// entry's row of u in key order).
struct WsLayout {
  size_t sched;      // 256 bytes: [0] the gemm kernel's block counter, [1] the union pass's CTA counter
  size_t k16;        // fp16 copy of k, [B, S_k + 1, 128]
  size_t binfo;      // int4 per block {tiles, dz scale exponent, entries, 0}
  size_t border;     // sparse: the blocks in descending tile count (processing order)
  size_t rec;        // sparse: tile records [nblocks][tcap][rstride bytes]
  size_t u;          // deterministic: per-entry dK rows [entries_cap][u_row_bytes(D)], in key order
  size_t hist;       // deterministic sparse: per-chunk key counts [nchunks, S_k] int32
  size_t key_start;  // deterministic: CSR offsets into u [B*S_k + 1] int32
  size_t total;
  long long nblocks;      // B * nbpb
  long long nchunks;      // deterministic sparse: B * ceil(nbpb / kSortBlocks)
  long long entries_cap;  // deterministic: rows of u
  int nbpb;               // blocks per batch, ceil(S_q / kBlkRows)
  int tcap;               // sparse: tile records per block, ceil(min(S_k, kBlkRows*L) / 128)
  int rstride;            // sparse: bytes per tile record (2560, or 3072 with positions)
};
WsLayout gemm_workspace_layout(int B, int S_q, int S_k, int H, int D, int L, int deterministic, int dense);

// The blocked gemm stage (blk.cu): fp16 copy of k, the union pass (sparse)
// or the scale pass (dense), the deterministic sort (det.cu), the gemm
// kernel (q by TMA, converted in place), the segment sum.
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st);

// Deterministic mode (det.cu): the key sort of the blocks' entries (sparse) or
// the closed-form CSR offsets (dense), run between the union pass and the
// gemm kernel; the segment sum after it.
cudaError_t launch_det_sort(const GemmArgs& a, const WsLayout& lay, cudaStream_t st);
cudaError_t launch_det_segsum(const GemmArgs& a, const WsLayout& lay, cudaStream_t st);

// fp16 copy of k into k16 ([B][S_k+1][128], zero padded, row S_k zero) that
// also zeroes nsched words of the counters at sched and nzero32 ints at
// zero32, and raises the fp16-range bit of *status for an entry outside the
// fp16 range.  pdl: launched programmatically behind this library's
// score-grad kernel.
cudaError_t launch_k_to_f16(const uint16_t* k, __half* k16, int B, int S_k, int D, unsigned* sched, int nsched,
                            unsigned* status, bool pdl, int num_sms, cudaStream_t st, int* zero32 = nullptr,
                            long long nzero32 = 0);

// The per-row gemm kernel (gemm.cu), atomic dK and no options: served to the
// allocation-free entry point, whose only scratch is its fp16 copy of k.
size_t rows_workspace_bytes(int B, int S_k);
cudaError_t prepare_gemm_rows();  // per device: the kernel's shared-memory attribute
cudaError_t launch_gemm_rows(const GemmArgs& a, cudaStream_t st);
// The per-row kernel alone on an fp16 copy of k made by the caller, its row
// counter zeroed by the caller; with select set it runs only when *select
// is 1 at its start (otherwise it exits at once).
cudaError_t launch_gemm_rows_kernel(const GemmArgs& a, const __half* k16, unsigned* counter, const unsigned* select,
                                    cudaStream_t st);

struct FwdArgs {
  const uint16_t* q;     // bf16 [rows, H, D]
  const uint16_t* k;     // bf16 [B, S_k, D]
  const float* w;        // [rows, H]
  const int32_t* idx;    // [rows, L] or nullptr (dense: key j of row t is valid iff j <= t)
  float* out;            // index_score [rows, L]
  int B, S_q, S_k, H, D, L;
  unsigned* status;
  int num_sms;
};
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t st);

}  // namespace ibwd
