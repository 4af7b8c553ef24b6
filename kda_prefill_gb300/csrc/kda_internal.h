// Internal interface between the host side of the C ABI (kda_api.cu) and the
// CUDA kernels (kda_kernels.cu).  Not installed; not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;  // K = V = head dimension
constexpr int kC = 64;   // tokens per chunk

// Everything one forward launch sequence needs.  Device pointers unless noted.
struct FwdParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g_raw;
    const float* beta_raw;
    __nv_bfloat16* out;
    int H;
    int N;
    int n_chunks;
    int64_t T;
    float lower_bound;

    // metadata (one int32 buffer uploaded by the host, see kda_api.cu)
    const int32_t* cu;         // [N+1] sequence bounds
    const int32_t* seq_off;    // [N+1] first chunk of each sequence
    const int32_t* chunk_seq;  // [n_chunks] sequence of each chunk
    const int32_t* chunk_tok;  // [n_chunks] first token of each chunk

    // workspace tiles, one set per (chunk, head), chunk-major
    float* ws_w;      // [n_chunks*H][C][D]   T (b k^ e^G)
    float* ws_qg;     // [n_chunks*H][C][D]   q^ e^G
    float* ws_kg;     // [n_chunks*H][C][D]   k^ e^{G_C - G}
    float* ws_u;      // [n_chunks*H][C][D]   T (b v)
    float* ws_aqk;    // [n_chunks*H][C][C]   decay-weighted q^ k^T, lower incl. diagonal
    float* ws_gamma;  // [n_chunks*H][D]      e^{G_C}

    // state (paged: st_in == st_out == pool, idx = state_indices;
    //        dense: separate bases, idx == nullptr means identity)
    const void* st_in;
    void* st_out;
    int64_t st_in_stride;   // elements between slots
    int64_t st_out_stride;
    const int32_t* st_in_idx;
    const int32_t* st_out_idx;
    const uint8_t* has_init;  // nullptr: every sequence has one iff st_in != nullptr
    int st_dtype;             // 0 fp32, 1 bf16, 2 fp16
};

// Workspace layout for an upper bound of chunks.
struct WsLayout {
    size_t off_w, off_qg, off_kg, off_u, off_aqk, off_gamma, total;
};
WsLayout workspace_layout(int64_t max_chunks, int H);

// Number of kernels one forward launches, and their names (launch order).
constexpr int kNumKernels = 2;
const char* kernel_name(int i);

// Enqueues the kernels of one forward on `s`.  When `marks` is non-null it
// holds kNumKernels + 1 events: marks[0] is recorded before the first kernel
// and marks[i + 1] after kernel i.
cudaError_t launch_forward(const FwdParams& p, cudaStream_t s, cudaEvent_t* marks);

}  // namespace kda
