// Host-side declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mla_decode.h"

namespace mla {

constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPage = 64;
constexpr int kHeadsPerCta = 64;
constexpr int kMaxSq = 16;

// Supported head counts: 16, 32, 48, 64 (one block) and 128 (two blocks).
inline bool heads_supported(int h) {
  return h == 16 || h == 32 || h == 48 || h == 64 || h == 128;
}
inline int head_blocks(int h) { return (h + kHeadsPerCta - 1) / kHeadsPerCta; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Records a failed CUDA call for mla_last_error(); returns MLA_ERR_CUDA.
int record_cuda_error(const char* where, cudaError_t e);
// Records a host-side validation failure (no CUDA error).
int record_error(const char* what, int status);

// Checks that `metadata` (device) matches the call; reads only the host-known
// sizes, never the device buffer.
int check_common(int batch, int s_q, int h_q, int num_sm_parts);

// Launches the split combine on `stream`; `pdl` enables programmatic
// dependent launch after the split kernel.
int launch_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                   const void* workspace, const float* attn_sink, void* out, float* lse,
                   cudaStream_t stream, bool pdl);

// Workspace partition: partial O then partial LSE.
inline int64_t workspace_rows(int batch, int s_q, int num_sm_parts) {
  return static_cast<int64_t>(batch) * s_q + num_sm_parts;
}

}  // namespace mla
