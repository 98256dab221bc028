// C-ABI front end of libcskv: synchronous argument checks, then launches (and the
// host staging copy of cskv_decode_layer).  Nothing here allocates device memory or
// synchronises (cskv_device_status excepted).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace cskv {

static std::atomic<unsigned long long> g_spin_limit{kDefaultSpinLimit};
unsigned long long spin_limit() { return g_spin_limit.load(std::memory_order_relaxed); }

static std::atomic<void*> g_ev_begin{nullptr}, g_ev_end{nullptr};
void timing_events(cudaEvent_t* begin, cudaEvent_t* end) {
  *begin = static_cast<cudaEvent_t>(g_ev_begin.load(std::memory_order_relaxed));
  *end = static_cast<cudaEvent_t>(g_ev_end.load(std::memory_order_relaxed));
}
void record_timing_event(cudaEvent_t ev, cudaStream_t stream) {
  if (ev == nullptr) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(stream, &cs);
  cudaEventRecordWithFlags(ev, stream,
                           cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

// Timing events go on a branch forked from the call's stream, so that each kernel
// on that stream still depends on the kernel before it alone (an event record
// between two kernels would keep a programmatic dependent launch from overlapping
// the kernel before it).  The branch joins the origin stream when the hook is
// turned off, which inside a stream capture must happen before the capture ends.
namespace {
struct TimingBranch {
  std::mutex mu;
  int device = -1;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaStream_t origin = nullptr;
  bool pending = false;
};
TimingBranch g_branch;

void branch_join_locked() {
  if (!g_branch.pending) return;
  cudaEventRecord(g_branch.join, g_branch.side);
  cudaStreamWaitEvent(g_branch.origin, g_branch.join, 0);
  g_branch.pending = false;
}

void branch_create_locked() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  if (g_branch.side != nullptr && g_branch.device == dev) return;
  if (g_branch.side != nullptr) {   // another device: the old helpers are dropped
    cudaStreamDestroy(g_branch.side);
    cudaEventDestroy(g_branch.fork);
    cudaEventDestroy(g_branch.join);
    g_branch.side = nullptr;
  }
  cudaStream_t st = nullptr;
  cudaEvent_t f = nullptr, j = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return;
  if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
    cudaStreamDestroy(st);
    if (f) cudaEventDestroy(f);
    return;
  }
  g_branch.side = st;
  g_branch.fork = f;
  g_branch.join = j;
  g_branch.device = dev;
}
}  // namespace

void record_timing_branch(cudaEvent_t ev, cudaStream_t stream) {
  if (ev == nullptr) return;
  std::lock_guard<std::mutex> lk(g_branch.mu);
  if (g_branch.side == nullptr || (g_branch.pending && g_branch.origin != stream)) {
    record_timing_event(ev, stream);
    return;
  }
  cudaEventRecord(g_branch.fork, stream);
  cudaStreamWaitEvent(g_branch.side, g_branch.fork, 0);
  record_timing_event(ev, g_branch.side);
  g_branch.origin = stream;
  g_branch.pending = true;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? CSKV_OK : CSKV_ERR_CUDA; }

// Checks a paged-cache descriptor for a lane of dimension `dim`; `formats` is a
// bit mask of the accepted cskv_format values.
static bool index_key_format(int fmt) {
  return fmt == CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT || fmt == CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT;
}

static bool paged_ok(const cskv_paged& c, int dim, unsigned formats) {
  if (c.pool == nullptr || !aligned(c.pool, 16)) return false;
  if (c.fmt < 0 || c.fmt > 4 || !((formats >> c.fmt) & 1u)) return false;
  if (c.dim != dim) return false;
  const size_t rb = cskv_row_bytes(c.fmt, c.dim);
  if (rb == 0) return false;
  if (c.page_bytes < static_cast<int64_t>(64 * rb) || c.page_bytes % 16 != 0) return false;
  if (c.num_pages <= 0) return false;
  if (c.block_table != nullptr && (c.max_pages <= 0 || !aligned(c.block_table, 4))) return false;
  return true;
}

// Host <-> device staging of a layer step's inputs and output.  Page-locked host
// memory is addressable from kernels on a unified-address system (over the coherent
// CPU-GPU link on Grace machines), so the copy runs on the SMs: a grid-stride loop of
// 16-byte loads and stores, one or two per thread, all in flight together, in place of a
// copy-engine transfer whose set-up dominates at a megabyte.  Other host memory is
// copied with cudaMemcpyAsync.
__global__ void __launch_bounds__(256) stage_copy_kernel(uint8_t* dst, const uint8_t* src, size_t n, int vec) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t t0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t n16 = vec ? n >> 4 : 0;
  for (size_t i = t0; i < n16; i += stride)
    reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
  for (size_t i = (n16 << 4) + t0; i < n; i += stride) dst[i] = src[i];
}

// The address a kernel uses for host pointer p, or nullptr if p is not page-locked.
static void* host_alias(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// n bytes from src to dst, one of them host memory (to_device: src is the host side).
static cudaError_t stage_copy(void* dst, const void* src, size_t n, bool to_device, cudaStream_t st) {
  void* alias = host_alias(to_device ? src : dst);
  if (alias == nullptr)
    return cudaMemcpyAsync(dst, src, n, to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost, st);
  uint8_t* d = static_cast<uint8_t*>(to_device ? dst : alias);
  const uint8_t* s = static_cast<const uint8_t*>(to_device ? alias : src);
  const int vec = aligned(d, 16) && aligned(s, 16);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t units = vec ? (n + 15) / 16 : n;
  const size_t want = (units + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < size_t(4) * sms ? want : size_t(4) * sms);
  stage_copy_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(d, s, n, vec);
  return cudaGetLastError();
}

}  // namespace cskv

using namespace cskv;

extern "C" {

size_t cskv_row_bytes(int32_t fmt, int32_t dim) {
  if (dim != 128 && dim != 512) return 0;
  switch (fmt) {
    case CSKV_FMT_BF16: return 2u * dim;
    case CSKV_FMT_FP8_E4M3_E8M0_B32: return dim + dim / 32;
    case CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT: return dim + 4;
    case CSKV_FMT_FP4_E2M1_E4M3_B16: return dim / 2 + dim / 16;
    case CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT: return dim == 128 ? dim / 2 + dim / 32 : 0;
    default: return 0;
  }
}

const char* cskv_status_string(int32_t s) {
  switch (s) {
    case CSKV_OK: return "ok";
    case CSKV_ERR_INVALID: return "invalid argument (nothing launched)";
    case CSKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSKV_ERR_CUDA: return "CUDA error";
    case CSKV_ERR_TIMEOUT: return "device wait timed out";
    case CSKV_ERR_BOUNDS: return "device index outside its table or pool";
    default: return "unknown status";
  }
}

int32_t cskv_version(void) { return 100; }

void cskv_set_spin_limit(uint64_t cycles) {
  g_spin_limit.store(cycles == 0 ? kDefaultSpinLimit : cycles, std::memory_order_relaxed);
}

void cskv_set_timing_events(void* begin, void* end) {
  const bool on = begin != nullptr && end != nullptr;
  {
    std::lock_guard<std::mutex> lk(g_branch.mu);
    branch_join_locked();
    if (on) branch_create_locked();
  }
  g_ev_begin.store(on ? begin : nullptr, std::memory_order_relaxed);
  g_ev_end.store(on ? end : nullptr, std::memory_order_relaxed);
}

int32_t cskv_rope_table(const int64_t* positions, int32_t n, double theta, double yarn_factor,
                        double yarn_original, double beta_fast, double beta_slow, float* out) {
  if (n < 0 || (n > 0 && (positions == nullptr || out == nullptr))) return CSKV_ERR_INVALID;
  if (!(theta > 1.0)) return CSKV_ERR_INVALID;
  const bool yarn = yarn_factor > 1.0;
  if (yarn && !(yarn_original > 0.0 && beta_fast > 0.0 && beta_slow > 0.0)) return CSKV_ERR_INVALID;
  constexpr int kPairs = 32, kRopeDim = 64;
  double f[kPairs];
  for (int k = 0; k < kPairs; ++k) f[k] = std::pow(theta, -2.0 * k / kRopeDim);
  if (yarn) {
    // the pair that turns `beta` times over the original length (the YaRN correction range)
    auto kb = [&](double beta) {
      return kRopeDim * std::log(yarn_original / (2.0 * M_PI * beta)) / (2.0 * std::log(theta));
    };
    const int lo = std::max(static_cast<int>(std::floor(kb(beta_fast))), 0);
    const int hi = std::min(static_cast<int>(std::ceil(kb(beta_slow))), kPairs - 1);
    const double span = std::max(static_cast<double>(hi - lo), 1e-3);
    for (int k = 0; k < kPairs; ++k) {
      const double ramp = std::min(std::max((k - lo) / span, 0.0), 1.0);
      f[k] = f[k] / yarn_factor * ramp + f[k] * (1.0 - ramp);
    }
  }
  for (int32_t i = 0; i < n; ++i) {
    const double p = static_cast<double>(positions[i]);
    for (int k = 0; k < kPairs; ++k) {
      const double a = p * f[k];
      out[(static_cast<size_t>(i) * kPairs + k) * 2 + 0] = static_cast<float>(std::cos(a));
      out[(static_cast<size_t>(i) * kPairs + k) * 2 + 1] = static_cast<float>(std::sin(a));
    }
  }
  return CSKV_OK;
}

int32_t cskv_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CSKV_ERR_CUDA;
  const unsigned int bits = take_err_compress() | take_err_index() | take_err_attention();
  if (bits & (1u << CSKV_ERR_TIMEOUT)) return CSKV_ERR_TIMEOUT;
  if (bits & (1u << CSKV_ERR_BOUNDS)) return CSKV_ERR_BOUNDS;
  if (bits) return CSKV_ERR_CUDA;
  return CSKV_OK;
}

int32_t cskv_encode_rows(const void* src, int32_t src_is_bf16, int32_t n, int32_t dim,
                         const int32_t* dst_req, const int32_t* dst_row, cskv_paged dst,
                         void* stream) {
  if (n < 0 || (dim != 128 && dim != 512)) return CSKV_ERR_INVALID;
  if (n > 0 && (src == nullptr || !aligned(src, 16))) return CSKV_ERR_INVALID;
  if (!paged_ok(dst, dim, 0x1Fu)) return CSKV_ERR_INVALID;
  if (index_key_format(dst.fmt) && dim != 128) return CSKV_ERR_INVALID;
  return cuda_status(launch_encode_rows(src, src_is_bf16 != 0, n, dim, dst_req, dst_row, dst,
                                        static_cast<int>(cskv_row_bytes(dst.fmt, dim)),
                                        static_cast<cudaStream_t>(stream)));
}

static int32_t compress_check(const void* kv, const void* gate, const void* prev_kv, const void* prev_gate,
                              const float* ape, const float* norm_w, float eps, const float* rope_cs,
                              int32_t S, int32_t T, int32_t ratio, int32_t overlap, int32_t dim,
                              const int32_t* req, const int32_t* first_entry, cskv_paged out) {
  if (kv == nullptr || gate == nullptr || req == nullptr || first_entry == nullptr)
    return CSKV_ERR_INVALID;
  if (dim != 128 && dim != 512) return CSKV_ERR_INVALID;
  if (S < 0 || T < 0 || ratio < 1 || ratio > 1024 || T % ratio != 0) return CSKV_ERR_INVALID;
  if (overlap != 0 && overlap != 1) return CSKV_ERR_INVALID;
  if (overlap && ratio > 8) return CSKV_ERR_INVALID;
  if ((prev_kv == nullptr) != (prev_gate == nullptr)) return CSKV_ERR_INVALID;
  if (!(eps >= 0.0f)) return CSKV_ERR_INVALID;
  if (!aligned(kv, 8) || !aligned(gate, 8) || (ape && !aligned(ape, 16))) return CSKV_ERR_INVALID;
  if (prev_kv && (!aligned(prev_kv, 8) || !aligned(prev_gate, 8))) return CSKV_ERR_INVALID;
  if ((norm_w && !aligned(norm_w, 16)) || (rope_cs && !aligned(rope_cs, 16))) return CSKV_ERR_INVALID;
  if (!paged_ok(out, dim, 0x1Fu)) return CSKV_ERR_INVALID;
  if (index_key_format(out.fmt) && dim != 128) return CSKV_ERR_INVALID;
  return CSKV_OK;
}

int32_t cskv_compress(const void* kv, const void* gate, const void* prev_kv, const void* prev_gate,
                      const float* ape, const float* norm_w, float eps, const float* rope_cs,
                      int32_t S, int32_t T, int32_t ratio, int32_t overlap, int32_t dim,
                      const int32_t* req, const int32_t* first_entry, cskv_paged out,
                      void* stream) {
  const int32_t st = compress_check(kv, gate, prev_kv, prev_gate, ape, norm_w, eps, rope_cs, S, T, ratio,
                                    overlap, dim, req, first_entry, out);
  if (st != CSKV_OK) return st;
  return cuda_status(launch_compress(kv, gate, prev_kv, prev_gate, ape, norm_w, eps, rope_cs, S, T,
                                     ratio, overlap, dim, req, first_entry, out,
                                     static_cast<int>(cskv_row_bytes(out.fmt, dim)),
                                     static_cast<cudaStream_t>(stream)));
}

static int32_t compress_many_check(const cskv_compress_job* jobs, int32_t njobs) {
  if (jobs == nullptr || njobs < 1 || njobs > 4) return CSKV_ERR_INVALID;
  for (int32_t j = 0; j < njobs; ++j) {
    const cskv_compress_job& q = jobs[j];
    const int32_t st = compress_check(q.kv, q.gate, q.prev_kv, q.prev_gate, q.ape, q.norm_w, q.eps, q.rope_cs,
                                      q.S, q.T, q.ratio, q.overlap, q.dim, q.req, q.first_entry, q.out);
    if (st != CSKV_OK) return st;
  }
  return CSKV_OK;
}

int32_t cskv_compress_many(const cskv_compress_job* jobs, int32_t njobs, void* stream) {
  const int32_t st = compress_many_check(jobs, njobs);
  if (st != CSKV_OK) return st;
  return cuda_status(launch_compress_many(jobs, njobs, static_cast<cudaStream_t>(stream)));
}

int32_t cskv_decode_append(const cskv_decode_job* jobs, int32_t njobs, const int32_t* pos, int32_t B,
                           void* stream) {
  if (jobs == nullptr || njobs < 1 || njobs > 8 || B < 0) return CSKV_ERR_INVALID;
  if (B > 0 && pos == nullptr) return CSKV_ERR_INVALID;
  for (int32_t j = 0; j < njobs; ++j) {
    const cskv_decode_job& q = jobs[j];
    if (q.kv == nullptr || (q.dim != 128 && q.dim != 512)) return CSKV_ERR_INVALID;
    if (q.ratio < 1 || q.ratio > 1024 || (q.overlap != 0 && q.overlap != 1)) return CSKV_ERR_INVALID;
    if (q.overlap && (q.ratio < 2 || q.ratio > 8)) return CSKV_ERR_INVALID;
    if (q.ring_rows < 0 || (q.ring_rows > 0 && q.ratio != 1)) return CSKV_ERR_INVALID;
    if (q.ratio > 1 && (q.gate == nullptr || q.state_kv == nullptr || q.state_gate == nullptr))
      return CSKV_ERR_INVALID;
    if (!(q.eps >= 0.0f)) return CSKV_ERR_INVALID;
    if (!aligned(q.kv, 8) || (q.gate && !aligned(q.gate, 8))) return CSKV_ERR_INVALID;
    if ((q.state_kv && !aligned(q.state_kv, 8)) || (q.state_gate && !aligned(q.state_gate, 8)))
      return CSKV_ERR_INVALID;
    if ((q.ape && !aligned(q.ape, 16)) || (q.norm_w && !aligned(q.norm_w, 16)) ||
        (q.rope_cs && !aligned(q.rope_cs, 16)))
      return CSKV_ERR_INVALID;
    if (!paged_ok(q.out, q.dim, 0x1Fu)) return CSKV_ERR_INVALID;
    if (index_key_format(q.out.fmt) && q.dim != 128) return CSKV_ERR_INVALID;
  }
  if (B == 0) return CSKV_OK;
  return cuda_status(launch_decode_append(jobs, njobs, pos, B, static_cast<cudaStream_t>(stream)));
}

size_t cskv_index_topk_workspace_size(int32_t B, int32_t max_ctx_len, int32_t ratio, int32_t Hi,
                                      int32_t k) {
  if (B <= 0 || max_ctx_len < 0 || ratio < 1 || Hi < 1 || k < 1) return 0;
  return index_workspace_bytes(B, max_ctx_len / ratio, Hi, k);
}

static int32_t index_check(const void* q_idx, const float* w, const cskv_paged& keys, const int32_t* ctx_len,
                           int32_t B, int32_t Hi, int32_t ratio, int32_t k, int32_t max_ctx_len,
                           const int32_t* topk_idx, const void* workspace, size_t workspace_bytes) {
  if (q_idx == nullptr || w == nullptr || ctx_len == nullptr || topk_idx == nullptr)
    return CSKV_ERR_INVALID;
  if (B < 1 || Hi < 1 || ratio < 1 || k < 1 || k > 2048 || max_ctx_len < 0) return CSKV_ERR_INVALID;
  if (Hi > 64) return CSKV_ERR_UNSUPPORTED;
  if (!aligned(q_idx, 16) || !aligned(w, 4)) return CSKV_ERR_INVALID;
  if (!paged_ok(keys, 128, (1u << CSKV_FMT_BF16) | (1u << CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT) |
                                 (1u << CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT)))
    return CSKV_ERR_INVALID;
  if (keys.block_table == nullptr) return CSKV_ERR_INVALID;
  const size_t need = index_workspace_bytes(B, max_ctx_len / ratio, Hi, k);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
    return CSKV_ERR_INVALID;
  return CSKV_OK;
}

int32_t cskv_index_topk(const void* q_idx, const float* w, cskv_paged keys, const int32_t* ctx_len,
                        int32_t B, int32_t Hi, int32_t ratio, int32_t k, int32_t max_ctx_len,
                        int32_t* topk_idx, float* topk_score, void* workspace,
                        size_t workspace_bytes, void* stream) {
  const int32_t st = index_check(q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len, topk_idx, workspace,
                                 workspace_bytes);
  if (st != CSKV_OK) return st;
  return cuda_status(launch_index_topk(q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len,
                                       topk_idx, topk_score, workspace,
                                       static_cast<cudaStream_t>(stream)));
}

int32_t cskv_index_topk_noalloc(const void* q_idx, const float* w, cskv_paged keys,
                                const int32_t* ctx_len, int32_t B, int32_t Hi, int32_t ratio,
                                int32_t k, int32_t max_ctx_len, int32_t* topk_idx, float* topk_score,
                                void* stream) {
  if (q_idx == nullptr || w == nullptr || ctx_len == nullptr || topk_idx == nullptr)
    return CSKV_ERR_INVALID;
  if (B < 1 || Hi < 1 || ratio < 1 || k < 1 || k > 2048 || max_ctx_len < 0) return CSKV_ERR_INVALID;
  if (Hi > 64) return CSKV_ERR_UNSUPPORTED;
  if (!aligned(q_idx, 16) || !aligned(w, 4)) return CSKV_ERR_INVALID;
  if (!paged_ok(keys, 128, (1u << CSKV_FMT_BF16) | (1u << CSKV_FMT_FP8_E4M3_ROWSCALE_PAGESPLIT) |
                                 (1u << CSKV_FMT_FP4_E2M1_E8M0_HADAMARD_PAGESPLIT)))
    return CSKV_ERR_INVALID;
  if (keys.block_table == nullptr) return CSKV_ERR_INVALID;
  // the whole workspace must fit in the library's fixed scratch array
  if (index_workspace_bytes(B, max_ctx_len / ratio, Hi, k) > CSKV_NOALLOC_SCRATCH_BYTES)
    return CSKV_ERR_INVALID;
  return cuda_status(launch_index_topk_noalloc(q_idx, w, keys, ctx_len, B, Hi, ratio, k, max_ctx_len,
                                               topk_idx, topk_score, static_cast<cudaStream_t>(stream)));
}

size_t cskv_sparse_decode_attn_workspace_size(int32_t B, int32_t H, int32_t max_ctx_len,
                                              int32_t ratio, int32_t k) {
  if (B <= 0 || H <= 0 || max_ctx_len < 0 || ratio < 1) return 0;
  return attn_workspace_bytes(B, H, max_ctx_len, ratio, k);
}

static int32_t attn_check(const void* q, const cskv_paged& main_kv, const void* swa, int32_t swa_fmt,
                          const int32_t* ctx_len, const int32_t* topk_idx, int32_t k, int32_t ratio,
                          int32_t max_ctx_len, float softmax_scale, const float* q_rope_cs, int32_t B,
                          int32_t H, const void* out, const void* workspace, size_t workspace_bytes) {
  if (q == nullptr || swa == nullptr || ctx_len == nullptr || q_rope_cs == nullptr || out == nullptr)
    return CSKV_ERR_INVALID;
  if (B < 1 || H < 1 || H > 128 || ratio < 1 || max_ctx_len < 0) return CSKV_ERR_INVALID;
  if (topk_idx != nullptr && (k < 1 || k > 2048)) return CSKV_ERR_INVALID;
  if (swa_fmt != CSKV_FMT_BF16 && swa_fmt != CSKV_FMT_FP8_E4M3_E8M0_B32) return CSKV_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(swa, 16) || !aligned(q_rope_cs, 16) || !aligned(out, 16))
    return CSKV_ERR_INVALID;
  if (!(softmax_scale > 0.0f)) return CSKV_ERR_INVALID;
  if (!paged_ok(main_kv, 512, (1u << CSKV_FMT_BF16) | (1u << CSKV_FMT_FP8_E4M3_E8M0_B32) |
                                  (1u << CSKV_FMT_FP4_E2M1_E4M3_B16)))
    return CSKV_ERR_INVALID;
  const size_t need = attn_workspace_bytes(B, H, max_ctx_len, ratio, topk_idx ? k : 0);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
    return CSKV_ERR_INVALID;
  return CSKV_OK;
}

int32_t cskv_sparse_decode_attn(const void* q, cskv_paged main_kv, const void* swa, int32_t swa_fmt,
                                const int32_t* ctx_len, const int32_t* topk_idx, int32_t k,
                                int32_t ratio, int32_t max_ctx_len, const float* sink,
                                float softmax_scale, const float* q_rope_cs, int32_t B, int32_t H,
                                void* out, void* workspace, size_t workspace_bytes, void* stream) {
  const int32_t st = attn_check(q, main_kv, swa, swa_fmt, ctx_len, topk_idx, k, ratio, max_ctx_len, softmax_scale,
                                q_rope_cs, B, H, out, workspace, workspace_bytes);
  if (st != CSKV_OK) return st;
  return cuda_status(launch_sparse_decode_attn(q, main_kv, swa, swa_fmt, ctx_len, topk_idx,
                                               topk_idx ? k : 0, ratio, max_ctx_len, sink,
                                               softmax_scale, q_rope_cs, B, H, out, workspace,
                                               static_cast<cudaStream_t>(stream)));
}

int32_t cskv_sparse_prefill_attn(const void* q, cskv_paged main_kv, cskv_paged window, const int32_t* req_of,
                                 const int32_t* pos1, const int32_t* topk_idx, int32_t k, int32_t ratio,
                                 int32_t max_ctx_len, const float* sink, float softmax_scale,
                                 const float* q_rope_cs, int32_t T, int32_t H, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (q == nullptr || pos1 == nullptr || q_rope_cs == nullptr || out == nullptr) return CSKV_ERR_INVALID;
  if (T < 1 || T > 65535 || H < 1 || H > 128 || ratio < 1 || max_ctx_len < 0) return CSKV_ERR_INVALID;
  if (topk_idx != nullptr && (k < 1 || k > 2048)) return CSKV_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(q_rope_cs, 16) || !aligned(out, 16)) return CSKV_ERR_INVALID;
  if (!(softmax_scale > 0.0f)) return CSKV_ERR_INVALID;
  if (!paged_ok(main_kv, 512, (1u << CSKV_FMT_BF16) | (1u << CSKV_FMT_FP8_E4M3_E8M0_B32) |
                                  (1u << CSKV_FMT_FP4_E2M1_E4M3_B16)))
    return CSKV_ERR_INVALID;
  if (!paged_ok(window, 512, (1u << CSKV_FMT_BF16) | (1u << CSKV_FMT_FP8_E4M3_E8M0_B32))) return CSKV_ERR_INVALID;
  const size_t need = attn_workspace_bytes(T, H, max_ctx_len, ratio, topk_idx ? k : 0);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return CSKV_ERR_INVALID;
  return cuda_status(launch_sparse_prefill_attn(q, main_kv, window, req_of, pos1, topk_idx, topk_idx ? k : 0,
                                                ratio, max_ctx_len, sink, softmax_scale, q_rope_cs, T, H, out,
                                                workspace, static_cast<cudaStream_t>(stream)));
}

int32_t cskv_decode_layer(const cskv_decode_layer_args* args, void* stream) {
  if (args == nullptr) return CSKV_ERR_INVALID;
  const cskv_decode_layer_args& a = *args;
  // every stage's arguments before anything is enqueued
  if (a.njobs < 0 || a.njobs > 4) return CSKV_ERR_INVALID;
  if (a.njobs > 0) {
    const int32_t st = compress_many_check(a.jobs, a.njobs);
    if (st != CSKV_OK) return st;
  }
  const bool csa = a.q_idx != nullptr;
  if (csa) {
    const int32_t st = index_check(a.q_idx, a.w, a.keys, a.ctx_len, a.B, a.Hi, a.ratio, a.k, a.max_ctx_len,
                                   a.topk_idx, a.index_workspace, a.index_workspace_bytes);
    if (st != CSKV_OK) return st;
  }
  {
    const int32_t st = attn_check(a.q, a.main_kv, a.swa, a.swa_fmt, a.ctx_len, csa ? a.topk_idx : nullptr, a.k,
                                  a.ratio, a.max_ctx_len, a.softmax_scale, a.q_rope_cs, a.B, a.H, a.out,
                                  a.attn_workspace, a.attn_workspace_bytes);
    if (st != CSKV_OK) return st;
  }
  if (a.in_bytes > 0 && (a.h_in == nullptr || a.d_in == nullptr)) return CSKV_ERR_INVALID;
  if (a.out_bytes > 0 && (a.h_out == nullptr || a.out_bytes > size_t(a.B) * a.H * 512 * 2)) return CSKV_ERR_INVALID;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // a job's per-step inputs (kv, gate, prev_*, rope_cs) in page-locked host memory are
  // read in place by the compressor through their device alias: it runs beside the
  // score kernel, whose tiles wait for it only at the step's newest entries
  cskv_compress_job jobs[4];
  for (int32_t j = 0; j < a.njobs; ++j) {
    jobs[j] = a.jobs[j];
    auto in_place = [](const void* p) -> const void* {
      const void* al = p != nullptr ? host_alias(p) : nullptr;
      return al != nullptr ? al : p;
    };
    jobs[j].kv = in_place(jobs[j].kv);
    jobs[j].gate = in_place(jobs[j].gate);
    jobs[j].prev_kv = in_place(jobs[j].prev_kv);
    jobs[j].prev_gate = in_place(jobs[j].prev_gate);
    jobs[j].rope_cs = static_cast<const float*>(in_place(jobs[j].rope_cs));
  }
  if (a.in_bytes > 0 && stage_copy(a.d_in, a.h_in, a.in_bytes, true, st) != cudaSuccess) return CSKV_ERR_CUDA;
  // CSA: the indexer's prep, the compressor and the score kernel overlap (the score kernel
  // waits for the compressor only before the tiles holding the index keys it writes),
  // and each request's attention starts as soon as its own selection is written
  const uint32_t* ready = nullptr;
  if (csa) {
    if (launch_index_topk_fused(a.q_idx, a.w, a.keys, a.ctx_len, a.B, a.Hi, a.ratio, a.k, a.max_ctx_len,
                                a.topk_idx, nullptr, a.index_workspace, jobs, a.njobs, st, &ready) != cudaSuccess)
      return CSKV_ERR_CUDA;
  } else if (a.njobs > 0 && launch_compress_many(jobs, a.njobs, st) != cudaSuccess) {
    return CSKV_ERR_CUDA;
  }
  const int32_t kk = csa ? a.k : 0;
  // a whole page-locked output buffer is written by the combine kernel itself, beside out;
  // page-locked host queries are read in place through their device alias
  void* out_alias = nullptr;
  if (a.out_bytes > 0 && a.out_bytes == size_t(a.B) * a.H * 512 * 2) out_alias = host_alias(a.h_out);
  const void* q_alias = host_alias(a.q);
  if (launch_sparse_decode_attn(q_alias != nullptr ? q_alias : a.q, a.main_kv, a.swa, a.swa_fmt, a.ctx_len, csa ? a.topk_idx : nullptr, kk,
                                a.ratio, a.max_ctx_len, a.sink, a.softmax_scale, a.q_rope_cs, a.B, a.H, a.out,
                                a.attn_workspace, st, out_alias, ready) != cudaSuccess)
    return CSKV_ERR_CUDA;
  if (a.out_bytes > 0 && out_alias == nullptr && stage_copy(a.h_out, a.out, a.out_bytes, false, st) != cudaSuccess)
    return CSKV_ERR_CUDA;
  return CSKV_OK;
}

}  // extern "C"
