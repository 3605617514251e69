// Device and host helpers shared by the gemm-stage kernels (the blocked
// kernel in blk_pipe.cuh and the per-row kernel in gemm.cu): scale helpers,
// the drain wait, the transposed dK reduction and the launch wrapper.
#pragma once
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ibwd {

// 2^e as a float, for |e| <= 126.
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// fp32 -> bf16 bits, round to nearest even (the optional bf16 outputs).
__device__ __forceinline__ uint16_t to_bf16(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exponent c of the power-of-two scale 2^c that puts m * 2^c in [2^13, 2^14):
// the largest |dz| then sits well inside the fp16 range.  0 when m is zero or
// not finite.
__device__ __forceinline__ int dz_scale_exponent(float m) {
  int c = 0;
  if (m > 0.f && m <= 3.0e38f) {
    int e;
    frexpf(m, &e);
    c = max(-120, min(120, 14 - e));
  }
  return c;
}

// A bounded wait on an mbarrier phase that ignores the abort flag: used only
// to drain work that was already issued before the kernel may exit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned* status, uint64_t limit_ns) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, status, limit_ns);
}

// One warp's share of a transposed dK tile: TMEM holds dK^T (lane = column d,
// TMEM column = tile entry), so after tcgen05.ld a warp holds its 32 columns
// of 32 entries in v.  It passes each half of the chunk through its own 2 KB
// of shared memory (16 entries x 32 floats) and reads it back four entries
// per instruction, so one 16-byte vector reduction per lane covers four
// 128-byte lines of four dK rows.  RED: red.global.add into base[ids[e]];
// otherwise plain stores (the deterministic mode's per-entry rows).
template <bool RED>
__device__ __forceinline__ void dk_chunk(float* base, const int* ids, const float (&v)[32], int nrow, float sc,
                                         int D, int dblk, float* stage) {
  const int lane = threadIdx.x & 31;
  const int rsub = lane >> 3, c4 = (lane & 7) * 4;  // this lane's entry in a group of four, column offset
  const bool con = dblk + c4 < D;                    // D % 8 == 0: the whole float4 is in range
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    if (hf * 16 >= nrow) break;  // uniform
    int idv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) idv[k] = ids[hf * 16 + rsub + 4 * k];
#pragma unroll
    for (int e = 0; e < 16; ++e) stage[e * 32 + lane] = v[hf * 16 + e] * sc;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = rsub + 4 * k;
      if (hf * 16 + e < nrow && con) {
        const float4 x = *reinterpret_cast<const float4*>(stage + e * 32 + c4);
        float* dst = base + (long long)idv[k] * D + dblk + c4;
        if (RED)
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(x.x), "f"(x.y), "f"(x.z),
                       "f"(x.w));
        else
          *reinterpret_cast<float4*>(dst) = x;
      }
    }
    __syncwarp();  // the stage is rewritten by the next half
  }
}

// The same for 32 entries read straight from TMEM, 16 columns at a time (half
// the live registers of dk_chunk), as fp32 reductions into base: ta
// addresses the warp's lane quarter at the chunk's first column; the ids are
// clamped to idmax, so every address stays inside the destination whatever a
// record holds.
__device__ __forceinline__ void dk_chunk_tmem(float* base, const int* ids, uint32_t ta, int nrow, float sc, int D,
                                              int dblk, float* stage, int idmax) {
  const int lane = threadIdx.x & 31;
  const int rsub = lane >> 3, c4 = (lane & 7) * 4;
  const bool con = dblk + c4 < D;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    if (hf * 16 >= nrow) break;  // uniform
    float v[16];
    tmem_ld16(ta + hf * 16, v);
    int idv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) idv[k] = min((unsigned)ids[hf * 16 + rsub + 4 * k], (unsigned)idmax);
    tmem_wait_ld_dep16(v);
#pragma unroll
    for (int e = 0; e < 16; ++e) stage[e * 32 + lane] = v[e] * sc;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = rsub + 4 * k;
      if (hf * 16 + e < nrow && con) {
        const float4 x = *reinterpret_cast<const float4*>(stage + e * 32 + c4);
        float* dst = base + (long long)idv[k] * D + dblk + c4;
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(x.x), "f"(x.y), "f"(x.z),
                     "f"(x.w));
      }
    }
    __syncwarp();  // the stage is rewritten by the next half
  }
}

// Exponent qe with max |q| < 2^qe, from the largest |q| of a block as bf16
// bits (the Q operand holds fp16, where magnitudes below 2^-25 are zero, so
// qe >= -24 covers every nonzero operand; non-finite q raises the range
// status and takes the top value).
__device__ __forceinline__ int q_exponent(unsigned bits) {
  if (bits == 0u) return 0;
  if (bits >= 0x7F80u) return 17;
  int e;
  frexpf(__uint_as_float(bits << 16), &e);
  return max(-24, min(17, e));
}

// The deterministic mode's form of dk_chunk_tmem: 32 entries' dK rows stored
// at their sorted positions as u rows (u_row_bytes(D) each: D fp16 values,
// each scaled by su, then the factor sector).  The warp that holds columns
// 0..31 (own_f) also writes each entry's factor sector: f and zeros, 32
// bytes from two lanes.  The caller picks su so that every value stays below
// 2^15.
__device__ __forceinline__ void dk_chunk_u16(char* u, const int* ids, uint32_t ta, int nrow, float su, float f, int D,
                                             int dblk, float* stage, int idmax, bool own_f) {
  const int lane = threadIdx.x & 31;
  const int rsub = lane >> 3, c4 = (lane & 7) * 4;
  const bool con = dblk + c4 < D;
  const int rb = u_row_bytes(D), fsec = rb - 32;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    if (hf * 16 >= nrow) break;  // uniform
    float v[16];
    tmem_ld16(ta + hf * 16, v);
    int idv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) idv[k] = min((unsigned)ids[hf * 16 + rsub + 4 * k], (unsigned)idmax);
    tmem_wait_ld_dep16(v);
#pragma unroll
    for (int e = 0; e < 16; ++e) stage[e * 32 + lane] = v[e] * su;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = rsub + 4 * k;
      if (hf * 16 + e < nrow) {
        char* row = u + (long long)idv[k] * rb;
        if (con) {
          const float4 x = *reinterpret_cast<const float4*>(stage + e * 32 + c4);
          const __half2 lo = __floats2half2_rn(x.x, x.y), hi = __floats2half2_rn(x.z, x.w);
          uint2 h;
          h.x = *reinterpret_cast<const uint32_t*>(&lo);
          h.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(row + 2 * (dblk + c4)) = h;
        }
        if (own_f && c4 < 8)
          *reinterpret_cast<uint4*>(row + fsec + 4 * c4) = make_uint4(c4 == 0 ? __float_as_uint(f) : 0u, 0u, 0u, 0u);
      }
    }
    __syncwarp();  // the stage is rewritten by the next half
  }
}

// Launch with programmatic stream serialization when pdl is set: the kernel
// may start before the previous one on the stream completes and must call
// griddep_wait() before reading what that one writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                      bool pdl, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace ibwd
