// Launchers and per-translation-unit error readers shared between the C-ABI
// front end (cskv_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/cskv.h"

namespace cskv {

// default bound of every mbarrier spin-wait, in SM cycles (about 1 s at 2 GHz)
constexpr unsigned long long kDefaultSpinLimit = 1ull << 31;
unsigned long long spin_limit();
// measurement hook around the indexer score kernel (may be null)
void timing_events(cudaEvent_t* begin, cudaEvent_t* end);
void record_timing_event(cudaEvent_t ev, cudaStream_t stream);
void record_timing_branch(cudaEvent_t ev, cudaStream_t stream);

cudaError_t launch_compress(const void* kv, const void* gate, const void* prev_kv,
                            const void* prev_gate, const float* ape, const float* norm_w, float eps,
                            const float* rope_cs, int S, int T, int ratio, int overlap, int dim,
                            const int32_t* req, const int32_t* first_entry, const cskv_paged& out,
                            int out_row_bytes, cudaStream_t stream);

cudaError_t launch_compress_many(const cskv_compress_job* jobs, int njobs, cudaStream_t stream,
                                 bool dependent = false);
cudaError_t launch_decode_append(const cskv_decode_job* jobs, int njobs, const int32_t* pos, int B,
                                 cudaStream_t stream);

cudaError_t launch_encode_rows(const void* src, int src_bf16, int n, int dim, const int32_t* req,
                               const int32_t* row, const cskv_paged& out, int out_row_bytes,
                               cudaStream_t stream);

size_t index_workspace_bytes(int B, int n_max, int Hi, int k);
cudaError_t launch_index_topk(const void* q_idx, const float* w, const cskv_paged& keys,
                              const int32_t* ctx_len, int B, int Hi, int ratio, int k,
                              int max_ctx_len, int32_t* topk_idx, float* topk_score,
                              void* workspace, cudaStream_t stream);

// One decode step's compressor and indexer, overlapped (cskv_decode_layer): the query
// prep, then compress_many(jobs) as a programmatic dependent of it, then the score
// kernel, which reads the index keys these jobs write only after they are complete.
// *ready receives the per-request flags that the selection raises (nullptr when the
// batch takes the cooperative large-batch kernel; the attention then waits for the
// whole indexer instead).
cudaError_t launch_index_topk_fused(const void* q_idx, const float* w, const cskv_paged& keys,
                                    const int32_t* ctx_len, int B, int Hi, int ratio, int k, int max_ctx_len,
                                    int32_t* topk_idx, float* topk_score, void* workspace,
                                    const cskv_compress_job* jobs, int njobs, cudaStream_t stream,
                                    const uint32_t** ready);

cudaError_t launch_index_topk_noalloc(const void* q_idx, const float* w, const cskv_paged& keys,
                                      const int32_t* ctx_len, int B, int Hi, int ratio, int k,
                                      int max_ctx_len, int32_t* topk_idx, float* topk_score,
                                      cudaStream_t stream);

size_t attn_workspace_bytes(int B, int H, int max_ctx, int ratio, int k);
cudaError_t launch_sparse_decode_attn(const void* q, const cskv_paged& kv, const void* swa, int swa_fmt,
                                      const int32_t* ctx_len, const int32_t* topk, int k, int ratio,
                                      int max_ctx, const float* sink, float softmax_scale,
                                      const float* q_rope, int B, int H, void* out, void* workspace,
                                      cudaStream_t stream, void* out_host = nullptr,
                                      const uint32_t* ready = nullptr);
cudaError_t launch_sparse_prefill_attn(const void* q, const cskv_paged& kv, const cskv_paged& win,
                                       const int32_t* req_of, const int32_t* pos1, const int32_t* topk, int k,
                                       int ratio, int max_ctx, const float* sink, float softmax_scale,
                                       const float* q_rope, int T, int H, void* out, void* workspace,
                                       cudaStream_t stream);

unsigned int take_err_compress();
unsigned int take_err_index();
unsigned int take_err_attention();

}  // namespace cskv
