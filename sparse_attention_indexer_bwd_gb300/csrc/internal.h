// Launchers shared between the translation units of libindexer_bwd.so.
// Each returns a cudaError_t from the launch (cudaSuccess when queued).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ibwd {

// Padded tile geometry of the gemm-stage kernel.
constexpr int kBM = 128;  // keys per tile (the MMA M dimension for Z and dK)
constexpr int kDP = 128;  // head dim padded to 128 (the MMA M dimension for dQ)
constexpr int kHP = 64;   // indexer heads padded to 64 (the MMA N dimension for Z and dQ)
constexpr int kSortRows = 8;  // query rows per chunk of the deterministic mode's key sort

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
};

struct WsLayout {
  size_t sched;      // the gemm kernel's row counter (one 256-byte block)
  size_t k16;        // fp16 copy of k, [B, S_k + 1, 128]
  size_t u;          // deterministic: per-slot dK rows [rows*L, D] fp32
  size_t hist;       // deterministic: per-chunk key counts [nchunks, S_k] int32
  size_t key_start;  // deterministic: CSR offsets [B*S_k + 1] int32
  size_t order;      // deterministic [rows*L] int32: position mode, each valid slot's position in key
                     // order (indexed by slot r*L + j); slot mode, the valid slots in key order
                     // (ascending (r, j) within a key)
  size_t total;
  long long nchunks;
};
WsLayout gemm_workspace_layout(int B, int S_q, int S_k, int H, int D, int L, int deterministic);

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st);
// Deterministic dK layout: true = dK rows in key order (positions staged with
// the rows), false = dK rows by slot, summed through a key-order slot list.
bool det_position_mode(const GemmArgs& a);

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
