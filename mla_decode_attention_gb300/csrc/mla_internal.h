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

// Host-side range checks of the size arguments shared by the decode entry
// points (the device buffer is never read here; the kernels compare the
// metadata header with the call themselves, see meta_header_matches).
int check_common(int batch, int s_q, int h_q, int num_sm_parts);

// Launches the split combine on `stream`; `pdl` enables programmatic
// dependent launch after the split kernel.
int launch_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                   const void* workspace, const float* attn_sink, void* out, float* lse,
                   cudaStream_t stream, bool pdl);

// Workspace partition: partial O [rows, h, 512] fp32, partial LSE [rows, h]
// fp32, then kWorkspaceCtrlBytes of control words.  Control word 0 holds the
// schedule the last split kernel on this workspace walked (0 = A, 1 = B, -1 =
// metadata rejected); the combine reads it, so the metadata itself is never
// written by a decode call.  Control word 1 is 0 when that schedule left the
// combine nothing to do (schedule B with every sequence non-empty: each one
// written by the split kernel), else 1.
constexpr int64_t kWorkspaceCtrlBytes = 64;
inline int64_t workspace_rows(int batch, int s_q, int num_sm_parts) {
  return static_cast<int64_t>(batch) * s_q + num_sm_parts;
}
inline int32_t* workspace_ctrl(void* workspace, int64_t rows_times_h) {
  return reinterpret_cast<int32_t*>(static_cast<float*>(workspace) + rows_times_h * (kDv + 1));
}
inline const int32_t* workspace_ctrl(const void* workspace, int64_t rows_times_h) {
  return reinterpret_cast<const int32_t*>(static_cast<const float*>(workspace) + rows_times_h * (kDv + 1));
}

}  // namespace mla
