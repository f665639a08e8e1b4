// C-ABI entry points of the MXFP4 sparse paged decode library (mx4sp.h).
//
// Host side only: argument validation in the style of the pages' own checks
// ("vllm.models.minimax_m3.amd.ops.mxfp4_pages", mxfp4_page_views: uint8 pages
// with a trailing 8704-byte contiguous axis, else an error; "vllm.models.
// minimax_m3.amd.mono.dispatch", _step_refusal: a reason string instead of a
// wrong result), the per-device status word, and the kernel launches.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace mx4 {
cudaError_t launch_insert(const float*, const float*, const float*, int64_t, int, const int64_t*,
                          uint8_t*, uint8_t*, int64_t, int64_t, uint8_t*, int64_t, int64_t,
                          uint32_t*, cudaStream_t);
cudaError_t launch_index_score(const uint16_t*, int, const uint8_t*, int64_t, int64_t,
                               const int32_t*, int, int64_t, const int32_t*, float*, int64_t,
                               uint32_t*, int, cudaStream_t);
cudaError_t launch_index_score_mxq(const uint16_t*, int, const uint8_t*, int64_t, int64_t,
                                   const int32_t*, int, int64_t, const int32_t*, float*, int64_t,
                                   uint32_t*, int, cudaStream_t);
cudaError_t launch_topk(const float*, int64_t, const int32_t*, int64_t, int, int, int32_t*,
                        void*, uint32_t*, int, cudaStream_t);
size_t topk_workspace_bytes(int64_t, int, int64_t);
cudaError_t launch_norm_rope_insert(const float*, const float*, const float*, const float*,
                                    const float*, int64_t, int, int, const int64_t*, const float*,
                                    int64_t, const float*, const float*, const float*,
                                    const float*, float, const int64_t*, uint8_t*, uint8_t*,
                                    int64_t, int64_t, uint8_t*, int64_t, int64_t, uint16_t*,
                                    uint16_t*, uint32_t*, cudaStream_t);
cudaError_t launch_decode(const uint16_t*, int64_t, int, const uint8_t*, const uint8_t*, int64_t,
                          int64_t, const int32_t*, int64_t, const int32_t*, const int32_t*, int,
                          float, float*, void*, uint32_t*, int, cudaStream_t);
size_t decode_workspace_bytes(int64_t, int, int);
cudaError_t launch_fp8_index_insert(const float*, int64_t, const int64_t*, float, uint8_t*,
                                    int64_t, int64_t, uint32_t*, cudaStream_t);
cudaError_t launch_index_score_fp8(const uint16_t*, int, const uint8_t*, int64_t, int64_t,
                                   const int32_t*, int, int64_t, const int32_t*, float, float*,
                                   int64_t, uint32_t*, int, cudaStream_t);
}  // namespace mx4

// Device status word: kernels OR MX4_STATUS_* bits into it when they skip bad
// data; mx4_check_status reads and clears it.
static __device__ uint32_t g_status;

namespace {

thread_local char g_err[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return MX4_OK;
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  uint32_t* status = nullptr;
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// Per-device set-up (first call on a device): the status word's device address
// and the SM count.  Done before any launch, outside stream capture.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MX4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MX4_ERR_UNSUPPORTED, "device id %d", dev);
  DeviceInfo& d = g_dev[dev];
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!d.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status);
    if (e != cudaSuccess)
      return fail(MX4_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
      return fail(MX4_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    d.status = static_cast<uint32_t*>(p);
    d.ready = true;
  }
  *out = &d;
  return MX4_OK;
}

// SM count of the current device, for sizes that depend on the grid; a large
// count (so a size on the safe side) when the device cannot be queried.
int current_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1024;
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(MX4_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return ok();
}


// Argument checks of sparse_paged_decode, shared by its allocation-free variant
// and by the whole-step call (the same rules, the caller's name in the reason):
// first the sizes and the geometry, then (after the caller's workspace check)
// the pointers.
int check_decode_sizes(const char* name, int64_t T, int q_per_seq, int H, int Hkv, int64_t B,
                       int k, float scale) {
  if (H != 16 || Hkv != 1)
    return fail(MX4_ERR_UNSUPPORTED,
                "%s: H = %d, Hkv = %d (supported: 16 query heads, 1 KV head)", name, H, Hkv);
  if (q_per_seq < 1 || q_per_seq > 8)
    return fail(MX4_ERR_UNSUPPORTED, "%s: q_per_seq = %d", name, q_per_seq);
  if (k < 1 || k > 65536) return fail(MX4_ERR_UNSUPPORTED, "%s: k = %d", name, k);
  if (B < 0 || T != B * q_per_seq) return fail(MX4_ERR_INVALID, "%s: T != B * q_per_seq", name);
  if (T > 0x7FFFFFFF / 8) return fail(MX4_ERR_UNSUPPORTED, "%s: T = %lld too large", name, (long long)T);
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(MX4_ERR_INVALID, "%s: scale is not finite", name);
  return MX4_OK;
}

int check_decode_pointers(const char* name, const uint16_t* q, const uint8_t* k_pages,
                          const uint8_t* v_pages, int64_t kv_page_stride, int64_t kv_head_stride,
                          int64_t num_pages, const int32_t* block_table, int64_t bt_width,
                          const int32_t* seq_lens, const int32_t* topk_idx, const float* out) {
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !topk_idx || !out)
    return fail(MX4_ERR_INVALID, "%s: NULL pointer", name);
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
      kv_page_stride % 16 || kv_head_stride % 16)
    return fail(MX4_ERR_INVALID, "%s: misaligned buffer or stride", name);
  if (num_pages < 1 || kv_page_stride < mx4::kPageBytes || bt_width < 1)
    return fail(MX4_ERR_INVALID, "%s: num_pages, page stride or bt_width", name);
  return MX4_OK;
}

// Shared by index_score and index_score_mxq: same arguments, same limits.
using ScoreLaunch = cudaError_t (*)(const uint16_t*, int, const uint8_t*, int64_t, int64_t,
                                    const int32_t*, int, int64_t, const int32_t*, float*, int64_t,
                                    uint32_t*, int, cudaStream_t);
int score_entry(const char* name, ScoreLaunch launch, const uint16_t* iq, int64_t T,
                int q_per_seq, const uint8_t* idx_pages, int64_t idx_page_stride,
                int64_t num_pages, const int32_t* block_table, int64_t B, int64_t bt_width,
                const int32_t* seq_lens, float* scores, int64_t ld_scores, void* stream) {
  if (q_per_seq < 1 || q_per_seq > 8)
    return fail(MX4_ERR_UNSUPPORTED, "%s: q_per_seq = %d (supported 1..8)", name, q_per_seq);
  if (B < 0 || B > 65535) return fail(MX4_ERR_UNSUPPORTED, "%s: B = %lld", name, (long long)B);
  if (T != B * q_per_seq)
    return fail(MX4_ERR_INVALID, "%s: T = %lld != B * q_per_seq", name, (long long)T);
  if (B == 0) return ok();
  if (!iq || !idx_pages || !block_table || !seq_lens || !scores)
    return fail(MX4_ERR_INVALID, "%s: NULL pointer", name);
  if (!aligned(iq, 16) || !aligned(idx_pages, 16) || idx_page_stride % 16 || !aligned(scores, 4))
    return fail(MX4_ERR_INVALID, "%s: misaligned iq, pages or page stride", name);
  if (num_pages < 1 || idx_page_stride < mx4::kPageBytes || bt_width < 1 || ld_scores < 1)
    return fail(MX4_ERR_INVALID, "%s: num_pages, page stride, bt_width or ld invalid", name);
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(launch(iq, q_per_seq, idx_pages, idx_page_stride, num_pages, block_table,
                            (int)B, bt_width, seq_lens, scores, ld_scores, d->status, d->num_sms,
                            static_cast<cudaStream_t>(stream)),
                     name);
}

}  // namespace

extern "C" {

const char* mx4_last_error(void) { return g_err; }

size_t mx4_page_bytes(void) { return (size_t)mx4::kPageBytes; }

int mx4_insert(const float* k, const float* v, const float* idx_k, int64_t T, int Hkv,
               const int64_t* slot_mapping, uint8_t* k_pages, uint8_t* v_pages,
               int64_t kv_page_stride, int64_t kv_head_stride, uint8_t* idx_pages,
               int64_t idx_page_stride, int64_t num_pages, void* stream) {
  if (T < 0) return fail(MX4_ERR_INVALID, "mx4_insert: T = %lld < 0", (long long)T);
  if (Hkv < 1 || Hkv > 8)
    return fail(MX4_ERR_UNSUPPORTED, "mx4_insert: Hkv = %d (supported 1..8)", Hkv);
  if (T == 0) return ok();
  if (!k || !v || !idx_k || !slot_mapping || !k_pages || !v_pages || !idx_pages)
    return fail(MX4_ERR_INVALID, "mx4_insert: NULL pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(idx_k, 16))
    return fail(MX4_ERR_INVALID, "mx4_insert: fp32 rows must be 16-byte aligned");
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(idx_pages, 16) ||
      kv_page_stride % 16 || kv_head_stride % 16 || idx_page_stride % 16)
    return fail(MX4_ERR_INVALID, "mx4_insert: pages must be 16-byte aligned with 16-byte strides");
  if (num_pages < 1 || kv_page_stride < mx4::kPageBytes || idx_page_stride < mx4::kPageBytes ||
      (Hkv > 1 && kv_head_stride < mx4::kPageBytes))
    return fail(MX4_ERR_INVALID, "mx4_insert: num_pages < 1 or a stride below 8704 bytes");
  if (T * (2 * Hkv + 1) > (int64_t)8 * 0x7FFFFFFF)
    return fail(MX4_ERR_UNSUPPORTED, "mx4_insert: T too large");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(mx4::launch_insert(k, v, idx_k, T, Hkv, slot_mapping, k_pages, v_pages,
                                        kv_page_stride, kv_head_stride, idx_pages,
                                        idx_page_stride, num_pages, d->status,
                                        static_cast<cudaStream_t>(stream)),
                     "mx4_insert");
}

int mx4_norm_rope_insert(const float* q, const float* iq, const float* k, const float* v,
                         const float* idx_k, int64_t T, int H, int Hkv, const int64_t* positions,
                         const float* cos_sin, int64_t max_pos, const float* g_q,
                         const float* g_k, const float* g_iq, const float* g_ik, float eps,
                         const int64_t* slot_mapping, uint8_t* k_pages, uint8_t* v_pages,
                         int64_t kv_page_stride, int64_t kv_head_stride, uint8_t* idx_pages,
                         int64_t idx_page_stride, int64_t num_pages, uint16_t* q_out,
                         uint16_t* iq_out, void* stream) {
  if (T < 0) return fail(MX4_ERR_INVALID, "mx4_norm_rope_insert: T = %lld < 0", (long long)T);
  if (H < 1 || H > 64 || Hkv < 1 || Hkv > 8)
    return fail(MX4_ERR_UNSUPPORTED, "mx4_norm_rope_insert: H = %d, Hkv = %d (1..64, 1..8)", H,
                Hkv);
  if (!(eps >= 0.f) || !(eps < INFINITY))
    return fail(MX4_ERR_INVALID, "mx4_norm_rope_insert: eps must be finite and >= 0");
  if (T == 0) return ok();
  if (!q || !iq || !k || !v || !idx_k || !positions || !cos_sin || !g_q || !g_k || !g_iq ||
      !g_ik || !slot_mapping || !k_pages || !v_pages || !idx_pages || !q_out || !iq_out)
    return fail(MX4_ERR_INVALID, "mx4_norm_rope_insert: NULL pointer");
  if (max_pos < 1) return fail(MX4_ERR_INVALID, "mx4_norm_rope_insert: max_pos < 1");
  if (!aligned(q, 16) || !aligned(iq, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(idx_k, 16) || !aligned(cos_sin, 16) || !aligned(g_q, 16) || !aligned(g_k, 16) ||
      !aligned(g_iq, 16) || !aligned(g_ik, 16) || !aligned(q_out, 8) || !aligned(iq_out, 8))
    return fail(MX4_ERR_INVALID, "mx4_norm_rope_insert: misaligned array");
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(idx_pages, 16) ||
      kv_page_stride % 16 || kv_head_stride % 16 || idx_page_stride % 16)
    return fail(MX4_ERR_INVALID,
                "mx4_norm_rope_insert: pages must be 16-byte aligned with 16-byte strides");
  if (num_pages < 1 || kv_page_stride < mx4::kPageBytes || idx_page_stride < mx4::kPageBytes ||
      (Hkv > 1 && kv_head_stride < mx4::kPageBytes))
    return fail(MX4_ERR_INVALID, "mx4_norm_rope_insert: num_pages < 1 or a stride below 8704");
  if (T * (H + 2 + 2 * Hkv) > (int64_t)8 * 0x7FFFFFFF)
    return fail(MX4_ERR_UNSUPPORTED, "mx4_norm_rope_insert: T too large");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(
      mx4::launch_norm_rope_insert(q, iq, k, v, idx_k, T, H, Hkv, positions, cos_sin, max_pos,
                                   g_q, g_k, g_iq, g_ik, eps, slot_mapping, k_pages, v_pages,
                                   kv_page_stride, kv_head_stride, idx_pages, idx_page_stride,
                                   num_pages, q_out, iq_out, d->status,
                                   static_cast<cudaStream_t>(stream)),
      "mx4_norm_rope_insert");
}

int index_score(const uint16_t* iq, int64_t T, int q_per_seq, const uint8_t* idx_pages,
                int64_t idx_page_stride, int64_t num_pages, const int32_t* block_table,
                int64_t B, int64_t bt_width, const int32_t* seq_lens, float* scores,
                int64_t ld_scores, void* stream) {
  return score_entry("index_score", mx4::launch_index_score, iq, T, q_per_seq, idx_pages,
                     idx_page_stride, num_pages, block_table, B, bt_width, seq_lens, scores,
                     ld_scores, stream);
}

int index_score_mxq(const uint16_t* iq, int64_t T, int q_per_seq, const uint8_t* idx_pages,
                    int64_t idx_page_stride, int64_t num_pages, const int32_t* block_table,
                    int64_t B, int64_t bt_width, const int32_t* seq_lens, float* scores,
                    int64_t ld_scores, void* stream) {
  // the tensor copy of the pool wants it 32-byte aligned with a page stride of 32s
  if (B > 0 && idx_pages && (!aligned(idx_pages, 32) || idx_page_stride % 32))
    return fail(MX4_ERR_INVALID, "index_score_mxq: index pages not 32-byte aligned or page "
                "stride not a multiple of 32");
  return score_entry("index_score_mxq", mx4::launch_index_score_mxq, iq, T, q_per_seq,
                     idx_pages, idx_page_stride, num_pages, block_table, B, bt_width, seq_lens,
                     scores, ld_scores, stream);
}

size_t index_topk_workspace(int64_t T, int k, int64_t ld_scores) {
  return mx4::topk_workspace_bytes(T, k, ld_scores);
}

int index_topk(const uint16_t* iq, int64_t T, int q_per_seq, const uint8_t* idx_pages,
               int64_t idx_page_stride, int64_t num_pages, const int32_t* block_table, int64_t B,
               int64_t bt_width, const int32_t* seq_lens, float* scores, int64_t ld_scores, int k,
               int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream) {
  static const char* kName = "index_topk";
  if (q_per_seq < 1 || q_per_seq > 8)
    return fail(MX4_ERR_UNSUPPORTED, "%s: q_per_seq = %d (supported 1..8)", kName, q_per_seq);
  if (k < 1 || k > 65536) return fail(MX4_ERR_UNSUPPORTED, "%s: k = %d", kName, k);
  if (B < 0 || B > 65535) return fail(MX4_ERR_UNSUPPORTED, "%s: B = %lld", kName, (long long)B);
  if (T != B * q_per_seq)
    return fail(MX4_ERR_INVALID, "%s: T = %lld != B * q_per_seq", kName, (long long)T);
  if (T > 65535) return fail(MX4_ERR_UNSUPPORTED, "%s: %lld tokens (max 65535)", kName, (long long)T);
  if (ld_scores < 1) return fail(MX4_ERR_INVALID, "%s: ld_scores < 1", kName);
  if ((ld_scores + 16383) / 16384 > 512)
    return fail(MX4_ERR_UNSUPPORTED, "%s: ld_scores = %lld (max 8388608)", kName,
                (long long)ld_scores);
  const size_t need = index_topk_workspace(T, k, ld_scores);
  if (ws_bytes < need)
    return fail(MX4_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", kName, ws_bytes, need);
  if (need > 0 && (!ws || !aligned(ws, 16)))
    return fail(MX4_ERR_INVALID, "%s: workspace NULL or not 16-byte aligned", kName);
  if (B == 0) return ok();
  if (!iq || !idx_pages || !block_table || !seq_lens || !scores || !topk_idx)
    return fail(MX4_ERR_INVALID, "%s: NULL pointer", kName);
  if (!aligned(iq, 16) || !aligned(idx_pages, 16) || idx_page_stride % 16 || !aligned(scores, 4))
    return fail(MX4_ERR_INVALID, "%s: misaligned iq, pages or page stride", kName);
  if (num_pages < 1 || idx_page_stride < mx4::kPageBytes || bt_width < 1)
    return fail(MX4_ERR_INVALID, "%s: num_pages, page stride or bt_width invalid", kName);
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = mx4::launch_index_score(iq, q_per_seq, idx_pages, idx_page_stride, num_pages,
                                          block_table, (int)B, bt_width, seq_lens, scores,
                                          ld_scores, d->status, d->num_sms, s);
  if (e == cudaSuccess)
    e = mx4::launch_topk(scores, ld_scores, seq_lens, T, q_per_seq, k, topk_idx,
                         need > 0 ? ws : nullptr, d->status, d->num_sms, s);
  return cuda_result(e, kName);
}

int fp8_index_insert(const float* idx_k, int64_t T, const int64_t* slot_mapping, float scale,
                     uint8_t* pages, int64_t page_stride, int64_t num_pages, void* stream) {
  if (T < 0) return fail(MX4_ERR_INVALID, "fp8_index_insert: T = %lld < 0", (long long)T);
  if (!(scale > 0.f) || !(scale < INFINITY))
    return fail(MX4_ERR_INVALID, "fp8_index_insert: scale must be finite and > 0");
  if (T == 0) return ok();
  if (!idx_k || !slot_mapping || !pages)
    return fail(MX4_ERR_INVALID, "fp8_index_insert: NULL pointer");
  if (!aligned(idx_k, 16) || !aligned(pages, 16) || page_stride % 16)
    return fail(MX4_ERR_INVALID, "fp8_index_insert: misaligned rows, pages or page stride");
  if (num_pages < 1 || page_stride < MX4_FP8_PAGE_BYTES)
    return fail(MX4_ERR_INVALID, "fp8_index_insert: num_pages < 1 or a stride below 16384");
  if (T > (int64_t)8 * 0x7FFFFFFF)
    return fail(MX4_ERR_UNSUPPORTED, "fp8_index_insert: T too large");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(mx4::launch_fp8_index_insert(idx_k, T, slot_mapping, scale, pages,
                                                  page_stride, num_pages, d->status,
                                                  static_cast<cudaStream_t>(stream)),
                     "fp8_index_insert");
}

int index_score_fp8(const uint16_t* iq, int64_t T, int q_per_seq, const uint8_t* pages,
                    int64_t page_stride, int64_t num_pages, const int32_t* block_table,
                    int64_t B, int64_t bt_width, const int32_t* seq_lens, float scale,
                    float* scores, int64_t ld_scores, void* stream) {
  if (q_per_seq < 1 || q_per_seq > 8)
    return fail(MX4_ERR_UNSUPPORTED, "index_score_fp8: q_per_seq = %d (supported 1..8)",
                q_per_seq);
  if (B < 0 || B > 65535)
    return fail(MX4_ERR_UNSUPPORTED, "index_score_fp8: B = %lld", (long long)B);
  if (T != B * q_per_seq)
    return fail(MX4_ERR_INVALID, "index_score_fp8: T = %lld != B * q_per_seq", (long long)T);
  if (!(scale > 0.f) || !(scale < INFINITY))
    return fail(MX4_ERR_INVALID, "index_score_fp8: scale must be finite and > 0");
  if (B == 0) return ok();
  if (!iq || !pages || !block_table || !seq_lens || !scores)
    return fail(MX4_ERR_INVALID, "index_score_fp8: NULL pointer");
  if (!aligned(iq, 16) || !aligned(pages, 16) || page_stride % 16 || !aligned(scores, 4))
    return fail(MX4_ERR_INVALID, "index_score_fp8: misaligned iq, pages or page stride");
  if (num_pages < 1 || page_stride < MX4_FP8_PAGE_BYTES || bt_width < 1 || ld_scores < 1)
    return fail(MX4_ERR_INVALID,
                "index_score_fp8: num_pages, page stride, bt_width or ld invalid");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(mx4::launch_index_score_fp8(iq, q_per_seq, pages, page_stride, num_pages,
                                                 block_table, (int)B, bt_width, seq_lens, scale,
                                                 scores, ld_scores, d->status, d->num_sms,
                                                 static_cast<cudaStream_t>(stream)),
                     "index_score_fp8");
}

size_t topk_select_workspace(int64_t T, int k, int64_t ld_scores) {
  return mx4::topk_workspace_bytes(T, k, ld_scores);
}

int topk_select(const float* scores, int64_t ld_scores, const int32_t* seq_lens, int64_t B,
                int q_per_seq, int k, int32_t* topk_idx, void* ws, size_t ws_bytes,
                void* stream) {
  if (q_per_seq < 1 || q_per_seq > 8)
    return fail(MX4_ERR_UNSUPPORTED, "topk_select: q_per_seq = %d (supported 1..8)", q_per_seq);
  if (k < 1 || k > 65536) return fail(MX4_ERR_UNSUPPORTED, "topk_select: k = %d", k);
  if (B < 0 || B * q_per_seq > 0x7FFFFFFF)
    return fail(MX4_ERR_INVALID, "topk_select: B = %lld", (long long)B);
  const int64_t T = B * q_per_seq;
  if (ld_scores < 1) return fail(MX4_ERR_INVALID, "topk_select: ld_scores < 1");
  if (T > 65535) return fail(MX4_ERR_UNSUPPORTED, "topk_select: %lld tokens (max 65535)", (long long)T);
  if ((ld_scores + 16383) / 16384 > 512)
    return fail(MX4_ERR_UNSUPPORTED, "topk_select: ld_scores = %lld (max 8388608)",
                (long long)ld_scores);
  const size_t need = topk_select_workspace(T, k, ld_scores);
  if (ws_bytes < need) return fail(MX4_ERR_WORKSPACE, "topk_select: workspace too small");
  if (need > 0 && (!ws || !aligned(ws, 16)))
    return fail(MX4_ERR_INVALID, "topk_select: workspace NULL or not 16-byte aligned");
  if (T == 0) return ok();
  if (!scores || !seq_lens || !topk_idx) return fail(MX4_ERR_INVALID, "topk_select: NULL pointer");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(mx4::launch_topk(scores, ld_scores, seq_lens, T, q_per_seq, k, topk_idx,
                                      need > 0 ? ws : nullptr, d->status, d->num_sms,
                                      static_cast<cudaStream_t>(stream)),
                     "topk_select");
}

size_t sparse_paged_decode_workspace(int64_t T, int k) {
  if (T < 0 || k < 1) return 0;
  return mx4::decode_workspace_bytes(T, k, current_sms());
}

int sparse_paged_decode(const uint16_t* q, int64_t T, int q_per_seq, int H, int Hkv,
                        const uint8_t* k_pages, const uint8_t* v_pages, int64_t kv_page_stride,
                        int64_t kv_head_stride, int64_t num_pages, const int32_t* block_table,
                        int64_t B, int64_t bt_width, const int32_t* seq_lens,
                        const int32_t* topk_idx, int k, float scale, float* out, void* ws,
                        size_t ws_bytes, void* stream) {
  static const char* kName = "sparse_paged_decode";
  if (int rc = check_decode_sizes(kName, T, q_per_seq, H, Hkv, B, k, scale)) return rc;
  if (ws_bytes < sparse_paged_decode_workspace(T, k))
    return fail(MX4_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", kName, ws_bytes,
                sparse_paged_decode_workspace(T, k));
  if (T == 0) return ok();
  if (int rc = check_decode_pointers(kName, q, k_pages, v_pages, kv_page_stride, kv_head_stride,
                                     num_pages, block_table, bt_width, seq_lens, topk_idx, out))
    return rc;
  if (!ws || !aligned(ws, 16)) return fail(MX4_ERR_INVALID, "%s: workspace NULL or misaligned", kName);
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  return cuda_result(mx4::launch_decode(q, T, q_per_seq, k_pages, v_pages, kv_page_stride,
                                        num_pages, block_table, bt_width, seq_lens, topk_idx, k,
                                        scale, out, ws, d->status, d->num_sms,
                                        static_cast<cudaStream_t>(stream)),
                     kName);
}

int mx4_check_status(void* stream, uint32_t* bits) {
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, d->status, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d->status, 0, sizeof h, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(MX4_ERR_CUDA, "mx4_check_status: %s", cudaGetErrorString(e));
  if (bits) *bits = h;
  if (h)
    return fail(MX4_ERR_BOUNDS, "kernels skipped bad data: status bits 0x%x%s%s%s%s%s", h,
                (h & MX4_STATUS_BAD_SLOT) ? " bad-slot" : "",
                (h & MX4_STATUS_BAD_PAGE) ? " bad-page" : "",
                (h & MX4_STATUS_BAD_LEN) ? " bad-seq-len" : "",
                (h & MX4_STATUS_BAD_INDEX) ? " bad-topk-index" : "",
                (h & MX4_STATUS_BAD_VALUE) ? " non-finite-input" : "");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// sparse_paged_decode_noalloc: sparse_paged_decode for callers that cannot
// allocate device memory.
//
// Some callers of this library have no way to obtain scratch memory: a host
// framework that owns every byte of device memory through its own pool and
// hands an extension only the operation's inputs and outputs, or a plain C or
// foreign-language runtime that can pass through buffers it was given but has
// no device allocator of its own.  For them this entry point keeps the split
// workspace in a fixed array of device memory that belongs to the library
// (every GPU that loads the library holds it until the process exits), so the
// call itself allocates nothing.
//
// The array's host-side name is not a device address, so its address is taken
// with cudaGetSymbolAddress once per device, by the first call on that device
// with the device current; make that first call before any stream capture.
// All calls on a device share the array: two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on it.  Nothing in
// it needs to start at zero -- the split kernel writes every (max, sum, output)
// entry it owns before the merge kernel reads it -- so the previous call's
// contents are harmless.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MX4_NOALLOC_SCRATCH_BYTES];

namespace {
void* g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mutex;

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MX4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MX4_ERR_UNSUPPORTED, "device id %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(MX4_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MX4_OK;
}
}  // namespace

extern "C" int sparse_paged_decode_noalloc(
    const uint16_t* q, int64_t T, int q_per_seq, int H, int Hkv, const uint8_t* k_pages,
    const uint8_t* v_pages, int64_t kv_page_stride, int64_t kv_head_stride, int64_t num_pages,
    const int32_t* block_table, int64_t B, int64_t bt_width, const int32_t* seq_lens,
    const int32_t* topk_idx, int k, float scale, float* out, void* stream) {
  static const char* kName = "sparse_paged_decode_noalloc";
  if (int rc = check_decode_sizes(kName, T, q_per_seq, H, Hkv, B, k, scale)) return rc;
  const size_t need = sparse_paged_decode_workspace(T, k);
  if (need > (size_t)MX4_NOALLOC_SCRATCH_BYTES)
    return fail(MX4_ERR_WORKSPACE,
                "%s: T = %lld, k = %d needs %zu bytes of scratch, more than the library's "
                "fixed %zu; use sparse_paged_decode with a caller workspace",
                kName, (long long)T, k, need, (size_t)MX4_NOALLOC_SCRATCH_BYTES);
  if (T == 0) return ok();
  if (int rc = check_decode_pointers(kName, q, k_pages, v_pages, kv_page_stride, kv_head_stride,
                                     num_pages, block_table, bt_width, seq_lens, topk_idx, out))
    return rc;
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  void* scratch = nullptr;
  if (int rc = noalloc_scratch(&scratch)) return rc;
  return cuda_result(mx4::launch_decode(q, T, q_per_seq, k_pages, v_pages, kv_page_stride,
                                        num_pages, block_table, bt_width, seq_lens, topk_idx, k,
                                        scale, out, scratch, d->status, d->num_sms,
                                        static_cast<cudaStream_t>(stream)),
                     kName);
}

// ---------------------------------------------------------------------------
// mx4_decode_step: one decode step from host memory to host memory.

namespace {
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

extern "C" void mx4_decode_step_input_offsets(int64_t T, int64_t n_new, size_t offsets[6]) {
  const size_t T_ = T > 0 ? (size_t)T : 0, n_ = n_new > 0 ? (size_t)n_new : 0;
  const size_t sizes[6] = {T_ * 16 * mx4::kHeadDim * 2, T_ * mx4::kHeadDim * 2,
                           n_ * mx4::kHeadDim * 4,      n_ * mx4::kHeadDim * 4,
                           n_ * mx4::kHeadDim * 4,      n_ * 8};
  size_t off = 0;
  for (int i = 0; i < 6; ++i) {
    offsets[i] = off;
    off += align256(sizes[i]);
  }
}

extern "C" size_t mx4_decode_step_input_bytes(int64_t T, int64_t n_new) {
  size_t off[6];
  mx4_decode_step_input_offsets(T, n_new, off);
  const size_t n_ = n_new > 0 ? (size_t)n_new : 0;
  return std::max<size_t>(256, off[5] + align256(n_ * 8));
}

namespace {

// The arguments of one decode step that stay the same from step to step.
struct StepCfg {
  int64_t n_new;
  uint8_t* k_pages;
  uint8_t* v_pages;
  int64_t kv_page_stride, kv_head_stride;
  uint8_t* idx_pages;
  int64_t idx_page_stride, num_pages;
  const int32_t* block_table;
  int64_t B, bt_width;
  const int32_t* seq_lens;
  int q_per_seq, k;
  float scale;
  float* d_scores;
  int64_t ld_scores;
  int32_t* d_topk_idx;
  void* topk_ws;
  size_t topk_ws_bytes;
  void* dec_ws;
  size_t dec_ws_bytes;
};

// Validation of a step whose packed inputs sit at `staging` (`staging_bytes`
// available) and whose output goes to d_out; nothing is enqueued.
int step_check(const char* name, const StepCfg& c, const void* staging, size_t staging_bytes,
               const float* d_out) {
  if (c.q_per_seq < 1 || c.q_per_seq > 8)
    return fail(MX4_ERR_UNSUPPORTED, "%s: q_per_seq = %d", name, c.q_per_seq);
  if (c.B < 0 || c.B > 65535)
    return fail(MX4_ERR_UNSUPPORTED, "%s: B = %lld", name, (long long)c.B);
  if (c.n_new < 0) return fail(MX4_ERR_INVALID, "%s: n_new < 0", name);
  const int64_t T = c.B * c.q_per_seq;
  const size_t in_bytes = mx4_decode_step_input_bytes(T, c.n_new);
  if (!staging) return fail(MX4_ERR_INVALID, "%s: NULL staging buffer", name);
  if (staging_bytes < in_bytes)
    return fail(MX4_ERR_WORKSPACE, "%s: staging %zu < %zu bytes", name, staging_bytes, in_bytes);
  if (!aligned(staging, 256))
    return fail(MX4_ERR_INVALID, "%s: staging buffer must be 256-byte aligned", name);
  size_t off[6];
  mx4_decode_step_input_offsets(T, c.n_new, off);
  const uint8_t* st = static_cast<const uint8_t*>(staging);
  if (int rc = check_decode_sizes(name, T, c.q_per_seq, 16, 1, c.B, c.k, c.scale)) return rc;
  if (T > 0)
    if (int rc = check_decode_pointers(
            name, reinterpret_cast<const uint16_t*>(st + off[0]), c.k_pages, c.v_pages,
            c.kv_page_stride, c.kv_head_stride, c.num_pages, c.block_table, c.bt_width,
            c.seq_lens, c.d_topk_idx, d_out))
      return rc;
  if (T > 65535 || (c.ld_scores + 16383) / 16384 > 512)
    return fail(MX4_ERR_UNSUPPORTED, "%s: T = %lld or ld_scores = %lld beyond topk_select's limits",
                name, (long long)T, (long long)c.ld_scores);
  if (!c.idx_pages || !c.d_scores || c.idx_page_stride % 16 || !aligned(c.idx_pages, 16) ||
      c.idx_page_stride < mx4::kPageBytes || c.ld_scores < 1)
    return fail(MX4_ERR_INVALID, "%s: index pages, page stride or scores", name);
  if (c.topk_ws_bytes < index_topk_workspace(T, c.k, c.ld_scores) ||
      c.dec_ws_bytes < sparse_paged_decode_workspace(T, c.k))
    return fail(MX4_ERR_WORKSPACE, "%s: a workspace is too small", name);
  return MX4_OK;
}

// The device part of a step whose packed inputs are already at `staging`:
// insert, score + select, decode into d_out, on `stream`.
int step_compute(const StepCfg& c, uint8_t* staging, float* d_out, void* stream) {
  const int64_t T = c.B * c.q_per_seq;
  size_t off[6];
  mx4_decode_step_input_offsets(T, c.n_new, off);
  const uint16_t* q = reinterpret_cast<const uint16_t*>(staging + off[0]);
  const uint16_t* iq = reinterpret_cast<const uint16_t*>(staging + off[1]);
  const float* k_new = reinterpret_cast<const float*>(staging + off[2]);
  const float* v_new = reinterpret_cast<const float*>(staging + off[3]);
  const float* idx_new = reinterpret_cast<const float*>(staging + off[4]);
  const int64_t* slots = reinterpret_cast<const int64_t*>(staging + off[5]);
  if (c.n_new > 0)
    if (int rc = mx4_insert(k_new, v_new, idx_new, c.n_new, 1, slots, c.k_pages, c.v_pages,
                            c.kv_page_stride, c.kv_head_stride, c.idx_pages, c.idx_page_stride,
                            c.num_pages, stream))
      return rc;
  if (int rc = index_topk(iq, T, c.q_per_seq, c.idx_pages, c.idx_page_stride, c.num_pages,
                          c.block_table, c.B, c.bt_width, c.seq_lens, c.d_scores, c.ld_scores,
                          c.k, c.d_topk_idx, c.topk_ws, c.topk_ws_bytes, stream))
    return rc;
  return sparse_paged_decode(q, T, c.q_per_seq, 16, 1, c.k_pages, c.v_pages, c.kv_page_stride,
                             c.kv_head_stride, c.num_pages, c.block_table, c.B, c.bt_width,
                             c.seq_lens, c.d_topk_idx, c.k, c.scale, d_out, c.dec_ws,
                             c.dec_ws_bytes, stream);
}

}  // namespace

extern "C" int mx4_decode_step(const void* h_inputs, int64_t n_new, void* d_staging,
                               size_t staging_bytes, uint8_t* k_pages, uint8_t* v_pages,
                               int64_t kv_page_stride, int64_t kv_head_stride,
                               uint8_t* idx_pages, int64_t idx_page_stride, int64_t num_pages,
                               const int32_t* block_table, int64_t B, int64_t bt_width,
                               const int32_t* seq_lens, int q_per_seq, int k, float scale,
                               float* d_scores, int64_t ld_scores, int32_t* d_topk_idx,
                               void* topk_ws, size_t topk_ws_bytes, void* dec_ws,
                               size_t dec_ws_bytes, float* d_out, float* h_out, void* stream) {
  static const char* kName = "mx4_decode_step";
  const StepCfg c{n_new,    k_pages,     v_pages,   kv_page_stride, kv_head_stride,
                  idx_pages, idx_page_stride, num_pages, block_table,   B,
                  bt_width, seq_lens,    q_per_seq, k,              scale,
                  d_scores, ld_scores,   d_topk_idx, topk_ws,       topk_ws_bytes,
                  dec_ws,   dec_ws_bytes};
  if (q_per_seq >= 1 && q_per_seq <= 8 && B == 0 && n_new == 0) return ok();
  if (!h_inputs || !h_out) return fail(MX4_ERR_INVALID, "%s: NULL pointer", kName);
  if (int rc = step_check(kName, c, d_staging, staging_bytes, d_out)) return rc;
  const int64_t T = B * q_per_seq;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(d_staging, h_inputs, mx4_decode_step_input_bytes(T, n_new),
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail(MX4_ERR_CUDA, "%s: input copy: %s", kName, cudaGetErrorString(e));
  if (int rc = step_compute(c, static_cast<uint8_t*>(d_staging), d_out, stream)) return rc;
  e = cudaMemcpyAsync(h_out, d_out, (size_t)T * 16 * mx4::kHeadDim * sizeof(float),
                      cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess)
    return fail(MX4_ERR_CUDA, "%s: output copy: %s", kName, cudaGetErrorString(e));
  return ok();
}

extern "C" int mx4_decode_steps(int64_t n_steps, const void* h_inputs, size_t h_inputs_stride,
                                int64_t n_new, void* d_staging, size_t staging_bytes,
                                uint8_t* k_pages, uint8_t* v_pages, int64_t kv_page_stride,
                                int64_t kv_head_stride, uint8_t* idx_pages,
                                int64_t idx_page_stride, int64_t num_pages,
                                const int32_t* block_table, int64_t B, int64_t bt_width,
                                const int32_t* seq_lens, int q_per_seq, int k, float scale,
                                float* d_scores, int64_t ld_scores, int32_t* d_topk_idx,
                                void* topk_ws, size_t topk_ws_bytes, void* dec_ws,
                                size_t dec_ws_bytes, float* d_out, float* h_out,
                                size_t h_out_stride, void* stream, void* h2d_stream,
                                void* d2h_stream) {
  static const char* kName = "mx4_decode_steps";
  const StepCfg c{n_new,    k_pages,     v_pages,   kv_page_stride, kv_head_stride,
                  idx_pages, idx_page_stride, num_pages, block_table,   B,
                  bt_width, seq_lens,    q_per_seq, k,              scale,
                  d_scores, ld_scores,   d_topk_idx, topk_ws,       topk_ws_bytes,
                  dec_ws,   dec_ws_bytes};
  if (n_steps < 0) return fail(MX4_ERR_INVALID, "%s: n_steps < 0", kName);
  if (n_steps == 0 || (q_per_seq >= 1 && q_per_seq <= 8 && B == 0 && n_new == 0)) return ok();
  if (!h_inputs || !h_out || !d_out) return fail(MX4_ERR_INVALID, "%s: NULL pointer", kName);
  if (!h2d_stream || !d2h_stream || stream == h2d_stream || stream == d2h_stream ||
      h2d_stream == d2h_stream)
    return fail(MX4_ERR_INVALID, "%s: two copy streams, not the default stream, distinct from "
                "each other and from the compute stream, are needed", kName);
  const int64_t T = B * q_per_seq;
  const size_t in_bytes = q_per_seq >= 1 && q_per_seq <= 8 && B >= 0 && n_new >= 0
                              ? mx4_decode_step_input_bytes(T, n_new)
                              : 0;
  const size_t set_bytes = align256(in_bytes);  // staging set b at d_staging + b * set_bytes
  if (staging_bytes < 2 * set_bytes)
    return fail(MX4_ERR_WORKSPACE, "%s: staging %zu < 2 x %zu bytes", kName, staging_bytes,
                set_bytes);
  uint8_t* stage[2] = {static_cast<uint8_t*>(d_staging),
                       static_cast<uint8_t*>(d_staging) + set_bytes};
  const size_t out_elems = (size_t)T * 16 * mx4::kHeadDim;
  float* out[2] = {d_out, d_out + out_elems};
  if (!aligned(out[1], 16)) return fail(MX4_ERR_INVALID, "%s: misaligned d_out", kName);
  for (int b = 0; b < 2; ++b)
    if (int rc = step_check(kName, c, stage[b], set_bytes, out[b])) return rc;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t hs = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ds = static_cast<cudaStream_t>(d2h_stream);
  // events: start, inputs_ready[2], compute_done[2], out_done[2]
  cudaEvent_t ev[7] = {};
  int made = 0;
  cudaError_t e = cudaSuccess;
  for (; made < 7 && e == cudaSuccess; ++made)
    e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
  auto release = [&]() {
    for (int i = 0; i < 7; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);  // released once the stream reaches them
  };
  if (e != cudaSuccess) {
    release();
    return fail(MX4_ERR_CUDA, "%s: event: %s", kName, cudaGetErrorString(e));
  }
  cudaEvent_t start = ev[0], *inputs_ready = ev + 1, *compute_done = ev + 3, *out_done = ev + 5;
  // the copies are ordered after the work already on `stream`
  e = cudaEventRecord(start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds, start, 0);
  int rc = MX4_OK;
  const uint8_t* hin = static_cast<const uint8_t*>(h_inputs);
  uint8_t* hout = reinterpret_cast<uint8_t*>(h_out);
  for (int64_t i = 0; i < n_steps && e == cudaSuccess && rc == MX4_OK; ++i) {
    const int b = (int)(i & 1);
    // step i's inputs into set b, once step i-2 has finished computing from it
    if (i >= 2) e = cudaStreamWaitEvent(hs, compute_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(stage[b], hin + (size_t)i * h_inputs_stride, in_bytes,
                          cudaMemcpyHostToDevice, hs);
    if (e == cudaSuccess) e = cudaEventRecord(inputs_ready[b], hs);
    // compute once the inputs are in and step i-2's output has been read back
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, inputs_ready[b], 0);
    if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(cs, out_done[b], 0);
    if (e != cudaSuccess) break;
    rc = step_compute(c, stage[b], out[b], stream);
    if (rc != MX4_OK) break;
    e = cudaEventRecord(compute_done[b], cs);
    // read step i's output back
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds, compute_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(hout + (size_t)i * h_out_stride, out[b], out_elems * sizeof(float),
                          cudaMemcpyDeviceToHost, ds);
    if (e == cudaSuccess) e = cudaEventRecord(out_done[b], ds);
  }
  // `stream` reaches the end of the call only after the last output copy (and so
  // after every copy of the call, both copy streams being in order)
  cudaError_t e2 = cudaEventRecord(start, ds);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(cs, start, 0);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(start, hs);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(cs, start, 0);
  release();
  if (rc != MX4_OK) return rc;
  if (e != cudaSuccess) return fail(MX4_ERR_CUDA, "%s: %s", kName, cudaGetErrorString(e));
  if (e2 != cudaSuccess) return fail(MX4_ERR_CUDA, "%s: %s", kName, cudaGetErrorString(e2));
  return ok();
}
