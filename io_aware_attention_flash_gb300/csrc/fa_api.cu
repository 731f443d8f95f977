// C ABI of libfa_gb300: argument validation, TMA descriptor creation and
// kernel launches.  See include/fa.h for the contract of every entry point.
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_kernels.cuh"
#include "ptx.cuh"

namespace {

// Device error word: kernels or-in kDevErr* bits; fa_get_device_error reads
// and clears it.
__device__ uint32_t g_fa_error_word;

// Limit of every bounded mbarrier wait in the attention kernels.  No wait of a
// correct launch comes near it; it only ends a wait that can never complete.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

using fa::kMaxDevices;

// Text of the last FA_ERR_CUDA on this host thread (fa_last_error_detail).
thread_local char t_detail[256] = "";

fa_status cuda_fail(const char* what, cudaError_t e) {
  snprintf(t_detail, sizeof(t_detail), "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
  return FA_ERR_CUDA;
}

// Device address of g_fa_error_word on the current device (cached per device).
fa_status error_word(uint32_t** out) {
  static uint32_t* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail("device ordinal out of range", cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fa_error_word);
    if (e != cudaSuccess || !p) return cuda_fail("cudaGetSymbolAddress(error word)", e);
    cache[dev] = static_cast<uint32_t*>(p);
  }
  *out = cache[dev];
  return FA_OK;
}

fa_status check_arch() {
  static int ok_cache[kMaxDevices] = {};  // 0 unknown, 1 ok, 2 wrong arch
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail("device ordinal out of range", cudaErrorInvalidDevice);
  if (ok_cache[dev] == 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", e);
    ok_cache[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return ok_cache[dev] == 1 ? FA_OK : FA_ERR_ARCH;
}

// Makes the device that owns `ptr` current on this host thread (binding its
// primary context, which the driver-API tensor-map encoder needs; a thread
// such as an autograd worker may have none bound yet) and checks that it is
// an sm_103 part.
fa_status bind_device(const void* ptr) {
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unregistered pointer
    return FA_ERR_NOT_DEVICE;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return FA_ERR_NOT_DEVICE;
  if ((e = cudaSetDevice(attr.device)) != cudaSuccess) return cuda_fail("cudaSetDevice", e);
  return check_arch();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bf16 tensor [outer, rows, H, d] (d innermost) viewed as a 4-D TMA map with a
// box_rows x 64-column box (128 rows for loads; 32 for the outputs O, dK and
// dV, which each warp stores for its own 32 rows) and 128-byte swizzle.  Rows past
// `rows` (within one outer index) read as zero and are not written.
fa_status make_map(CUtensorMap* map, const void* ptr, int d, int H, long long rows, int outer,
                   int box_rows = fa::kTile) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled entry point not found", cudaErrorSymbolNotFound);
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                                 static_cast<cuuint64_t>(rows) * H * d * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(t_detail, sizeof(t_detail), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// fp32 dQ accumulator [rows, H, d] as a 3-D TMA map (d, H, rows) with a
// 32-column x 32-row box and 128-byte swizzle: the target of the backward's
// bulk reduce-adds.  Rows past `rows` are clipped.
fa_status make_map_dq(CUtensorMap* map, const void* ptr, int d, int H, long long rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cuda_fail("cuTensorMapEncodeTiled entry point not found", cudaErrorSymbolNotFound);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(H) * d * 4};
  const cuuint32_t box[3] = {32, 1, 32};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(t_detail, sizeof(t_detail), "cuTensorMapEncodeTiled (dQ accumulator) failed (CUresult %d)",
             static_cast<int>(r));
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// One-shot kernel timing hook of the calling host thread (fa_set_kernel_events).
thread_local cudaEvent_t t_main_start = nullptr;
thread_local cudaEvent_t t_main_end = nullptr;

size_t pad256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Shape limits: int32 row indices, and one CTA per (sequence, head, tile)
// within the one-dimensional grid's 2^31 - 1 blocks.
fa_status check_common(int H, int d, float scale) {
  if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
  if (H <= 0 || H > 65535) return FA_ERR_SHAPE;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  return FA_OK;
}

fa_status check_rows(long long nseq, long long rows, long long max_seqlen, int H, int d) {
  if (nseq <= 0 || rows <= 0 || max_seqlen <= 0) return FA_ERR_SHAPE;
  if (rows > 0x7fffffffLL || nseq * H > 0x7fffffffLL) return FA_ERR_SHAPE;
  if (rows * H * static_cast<long long>(d) > (1LL << 40)) return FA_ERR_SHAPE;
  if (nseq * H * ((max_seqlen + fa::kTile - 1) / fa::kTile) > 0x7fffffffLL) return FA_ERR_SHAPE;
  return FA_OK;
}

#define FA_TRY(expr)                 \
  do {                               \
    const fa_status _st = (expr);    \
    if (_st != FA_OK) return _st;    \
  } while (0)

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu, int nseq,
                   int max_seqlen, long long rows_per_outer, int outer, int H, int d, float scale, int causal,
                   void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGN;
  FA_TRY(bind_device(q));
  uint32_t* err = nullptr;
  FA_TRY(error_word(&err));
  CUtensorMap tq, tk, tv, to;
  FA_TRY(make_map(&tq, q, d, H, rows_per_outer, outer));
  FA_TRY(make_map(&tk, k, d, H, rows_per_outer, outer));
  FA_TRY(make_map(&tv, v, d, H, rows_per_outer, outer));
  FA_TRY(make_map(&to, o, d, H, rows_per_outer, outer, 32));
  fa::FwdParams p{};
  p.sv.cu_seqlens = cu;
  p.sv.H = H;
  p.sv.N = static_cast<int>(rows_per_outer);
  p.sv.lse_stride = cu ? max_seqlen : static_cast<int>(rows_per_outer);
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.scale_log2 = scale * fa::kLog2e;
  p.causal = causal ? 1 : 0;
  p.err = err;
  p.timeout_ns = kWaitLimitNs;
  const cudaError_t e = fa::launch_fwd(d, tq, tk, tv, to, p, nseq, max_seqlen, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("forward launch", e);
}

// D (fp32, stat_elems) then the fp32 dQ accumulator, tiled by 128 rows (rows
// rounded up to a multiple of 128).
size_t bwd_ws_bytes(long long stat_elems, long long rows, int H, int d) {
  const size_t rows128 = static_cast<size_t>((rows + fa::kTile - 1) / fa::kTile) * fa::kTile;
  return pad256(static_cast<size_t>(stat_elems) * 4) + rows128 * H * d * 4;
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, const int* cu, int nseq, int max_seqlen,
                   long long rows_per_outer, int outer, int H, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGN;
  const long long rows = rows_per_outer * outer;
  const long long stat_elems = static_cast<long long>(nseq) * H * (cu ? max_seqlen : rows_per_outer);
  if (!ws || ws_bytes < bwd_ws_bytes(stat_elems, rows, H, d)) return FA_ERR_WORKSPACE;
  if (!aligned16(ws)) return FA_ERR_ALIGN;
  FA_TRY(bind_device(q));
  uint32_t* err = nullptr;
  FA_TRY(error_word(&err));
  CUtensorMap tq, tk, tv, tdo;
  FA_TRY(make_map(&tq, q, d, H, rows_per_outer, outer));
  FA_TRY(make_map(&tk, k, d, H, rows_per_outer, outer));
  FA_TRY(make_map(&tv, v, d, H, rows_per_outer, outer));
  FA_TRY(make_map(&tdo, dout, d, H, rows_per_outer, outer));
  fa::BwdParams p{};
  p.sv.cu_seqlens = cu;
  p.sv.H = H;
  p.sv.N = static_cast<int>(rows_per_outer);
  p.sv.lse_stride = cu ? max_seqlen : static_cast<int>(rows_per_outer);
  p.o = static_cast<const uint16_t*>(o);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.dpsum = static_cast<float*>(ws);
  p.dq_accum = reinterpret_cast<float*>(static_cast<char*>(ws) + pad256(static_cast<size_t>(stat_elems) * 4));
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.scale = scale;
  p.scale_log2 = scale * fa::kLog2e;
  p.causal = causal ? 1 : 0;
  p.rows = static_cast<int>(rows);
  p.nseq = nseq;
  p.err = err;
  p.timeout_ns = kWaitLimitNs;
  CUtensorMap tdq, tdk, tdv;
  FA_TRY(make_map_dq(&tdq, p.dq_accum, d, H, rows));
  FA_TRY(make_map(&tdk, dk, d, H, rows_per_outer, outer, 32));
  FA_TRY(make_map(&tdv, dv, d, H, rows_per_outer, outer, 32));
  cudaEvent_t ev0 = t_main_start, ev1 = t_main_end;
  t_main_start = t_main_end = nullptr;
  const cudaError_t e =
      fa::launch_bwd(d, tq, tk, tv, tdo, tdq, tdk, tdv, p, max_seqlen, static_cast<cudaStream_t>(stream), ev0, ev1);
  return e == cudaSuccess ? FA_OK : cuda_fail("backward launch", e);
}

// One CTA waits on an mbarrier that nothing arrives on, with a short limit.
__global__ void fa_wait_timeout_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t barrier;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(fa::smem_u32(&barrier), 1);
    fa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) fa::wait_bounded(fa::smem_u32(&barrier), 0, &abort_flag, err, limit_ns);
  __syncthreads();
}

// Split-KV decode: keys per split and number of splits.  A split is 1 to 8
// key tiles, sized so that there are about kDecodeTargetItems work items
// where the cache allows.  The choice depends only on the shapes (not on the
// device), so the workspace size does too; the persistent split kernel's grid
// is sized from the SM count of the device it runs on.  608 is four items per
// SM of a 152-SM part; on a part with a different SM count only the balance
// of items over SMs changes, not the result.
constexpr long long kDecodeTargetItems = 608;

void decode_split(int B, int H, int Nk, int* splits, int* split_len) {
  constexpr long long kTargetItems = kDecodeTargetItems;
  const long long tiles = (Nk + fa::kTile - 1) / fa::kTile;
  long long per = (tiles * B * H + kTargetItems - 1) / kTargetItems;
  per = per < 1 ? 1 : (per > 8 ? 8 : per);
  *split_len = static_cast<int>(per * fa::kTile);
  *splits = static_cast<int>((Nk + *split_len - 1) / *split_len);
}

size_t decode_ws_bytes(int B, int H, int Nq, int Nk, int d) {
  int splits = 0, split_len = 0;
  decode_split(B, H, Nk, &splits, &split_len);
  const size_t parts = static_cast<size_t>(B) * H * splits * Nq;
  return pad256(parts * d * 4) + pad256(parts * 2 * 4);
}

fa_status check_decode(int B, int H, int Nq, int Nk, int d, float scale) {
  FA_TRY(check_common(H, d, scale));
  if (B <= 0 || Nq <= 0 || Nq > 8 || Nk <= 0) return FA_ERR_SHAPE;
  FA_TRY(check_rows(B, static_cast<long long>(B) * Nk, Nk, H, d));
  if (static_cast<long long>(B) * H * Nq > (1LL << 31) / 32) return FA_ERR_SHAPE;
  return FA_OK;
}

}  // namespace

namespace fa {
cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
  fa_wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}
}  // namespace fa

extern "C" {

FA_API const char* fa_status_string(fa_status status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "null pointer argument";
    case FA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FA_ERR_HEAD_DIM: return "head dim must be 64 or 128";
    case FA_ERR_SHAPE: return "shape out of range";
    case FA_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case FA_ERR_CUDA: return "CUDA runtime or launch failure";
    case FA_ERR_TIMEOUT: return "device wait timed out; outputs invalid";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_SCALE: return "scale is not finite";
    case FA_ERR_NOT_DEVICE: return "q is not a device pointer";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the static no-alloc array holds";
    default: return "unknown status";
  }
}

FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                        float scale, int causal, void* stream) {
  FA_TRY(check_common(H, d, scale));
  if (B <= 0 || N <= 0) return FA_ERR_SHAPE;
  FA_TRY(check_rows(B, static_cast<long long>(B) * N, N, H, d));
  return fwd_impl(q, k, v, o, lse, nullptr, B, N, N, B, H, d, scale, causal, stream);
}

FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  return bwd_ws_bytes(static_cast<long long>(B) * H * N, static_cast<long long>(B) * N, H, d);
}

FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        int B, int H, int N, int d, float scale, int causal, void* stream) {
  FA_TRY(check_common(H, d, scale));
  if (B <= 0 || N <= 0) return FA_ERR_SHAPE;
  FA_TRY(check_rows(B, static_cast<long long>(B) * N, N, H, d));
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, nullptr, B, N, N, B, H, d, scale,
                  causal, stream);
}

FA_API fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int* cu_seqlens, int nseq, int max_seqlen, int total, int H, int d, float scale,
                               int causal, void* stream) {
  FA_TRY(check_common(H, d, scale));
  if (!cu_seqlens) return FA_ERR_NULL;
  FA_TRY(check_rows(nseq, total, max_seqlen, H, d));
  return fwd_impl(q, k, v, o, lse, cu_seqlens, nseq, max_seqlen, total, 1, H, d, scale, causal, stream);
}

FA_API size_t fa_bwd_varlen_workspace_bytes(int total, int nseq, int max_seqlen, int H, int d) {
  if (total <= 0 || nseq <= 0 || max_seqlen <= 0 || H <= 0 || d <= 0) return 0;
  return bwd_ws_bytes(static_cast<long long>(nseq) * H * max_seqlen, total, H, d);
}

FA_API fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, void* workspace,
                               size_t workspace_bytes, const int* cu_seqlens, int nseq, int max_seqlen, int total,
                               int H, int d, float scale, int causal, void* stream) {
  FA_TRY(check_common(H, d, scale));
  if (!cu_seqlens) return FA_ERR_NULL;
  FA_TRY(check_rows(nseq, total, max_seqlen, H, d));
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, cu_seqlens, nseq, max_seqlen, total,
                  1, H, d, scale, causal, stream);
}

FA_API size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (check_decode(B, H, Nq, Nk, d, 1.0f) != FA_OK) return 0;
  return decode_ws_bytes(B, H, Nq, Nk, d);
}

FA_API fa_status fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                               size_t workspace_bytes, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                               void* stream) {
  FA_TRY(check_decode(B, H, Nq, Nk, d, scale));
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
    return FA_ERR_ALIGN;
  if (workspace_bytes < decode_ws_bytes(B, H, Nq, Nk, d)) return FA_ERR_WORKSPACE;
  FA_TRY(bind_device(q));
  uint32_t* err = nullptr;
  FA_TRY(error_word(&err));
  CUtensorMap tk, tv;
  FA_TRY(make_map(&tk, k, d, H, Nk, B));
  FA_TRY(make_map(&tv, v, d, H, Nk, B));
  fa::DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  decode_split(B, H, Nk, &p.splits, &p.split_len);
  const size_t parts = static_cast<size_t>(B) * H * p.splits * Nq;
  p.o_part = static_cast<float*>(workspace);
  p.ml_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + pad256(parts * d * 4));
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.scale_log2 = scale * fa::kLog2e;
  p.causal = causal ? 1 : 0;
  p.err = err;
  p.timeout_ns = kWaitLimitNs;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail("device query", e);
  const long long items = static_cast<long long>(B) * H * p.splits;
  const int grid = static_cast<int>(items < sms ? items : sms);
  e = fa::launch_decode(d, tk, tv, p, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("decode launch", e);
}

FA_API fa_status fa_get_device_error(void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  // The error word of the device the stream belongs to (the legacy default
  // stream belongs to the current device); the caller's current device is
  // restored afterwards.
  int cur = 0, dev = 0;
  if ((e = cudaGetDevice(&cur)) != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if ((e = cudaStreamGetDevice(s, &dev)) != cudaSuccess) return cuda_fail("cudaStreamGetDevice", e);
  if (dev != cur && (e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail("cudaSetDevice", e);
  uint32_t word = 0;
  fa_status st = FA_OK;
  if ((e = cudaMemcpyFromSymbol(&word, g_fa_error_word, sizeof(word))) != cudaSuccess) {
    st = cuda_fail("read error word", e);
  } else if (word != 0) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpyToSymbol(g_fa_error_word, &zero, sizeof(zero))) != cudaSuccess) {
      st = cuda_fail("clear error word", e);
    } else if (word & fa::kDevErrTimeout) {
      st = FA_ERR_TIMEOUT;
    } else {
      snprintf(t_detail, sizeof(t_detail), "device error word 0x%x", word);
      st = FA_ERR_CUDA;
    }
  }
  if (dev != cur) {
    e = cudaSetDevice(cur);
    if (st == FA_OK && e != cudaSuccess) st = cuda_fail("cudaSetDevice (restore)", e);
  }
  return st;
}

FA_API const char* fa_last_error_detail(void) { return t_detail; }

}  // extern "C"

namespace {

// Scratch of fa_bwd_noalloc: D and the fp32 dQ accumulator for callers that
// cannot hand the library a workspace.  File-scope static device storage:
// every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the array's name is only a host-side stand-in,
// so kernels must be given this address, never the name.
fa_status noalloc_scratch(void** out) {
  static void* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail("device ordinal out of range", cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail("cudaGetSymbolAddress(no-alloc scratch)", e);
    cache[dev] = p;
  }
  *out = cache[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

FA_API fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                float scale, int causal, void* stream) {
  FA_TRY(check_common(H, d, scale));
  if (B <= 0 || N <= 0) return FA_ERR_SHAPE;
  FA_TRY(check_rows(B, static_cast<long long>(B) * N, N, H, d));
  const size_t need = bwd_ws_bytes(static_cast<long long>(B) * H * N, static_cast<long long>(B) * N, H, d);
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  if (!q) return FA_ERR_NULL;
  FA_TRY(bind_device(q));  // the scratch address is per device: look it up with q's device current
  void* scratch = nullptr;
  FA_TRY(noalloc_scratch(&scratch));
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, scratch, FA_NOALLOC_SCRATCH_BYTES, nullptr, B, N, N, B, H, d,
                  scale, causal, stream);
}

FA_API fa_status fa_set_kernel_events(void* start_event, void* end_event) {
  if ((start_event == nullptr) != (end_event == nullptr)) return FA_ERR_NULL;
  t_main_start = static_cast<cudaEvent_t>(start_event);
  t_main_end = static_cast<cudaEvent_t>(end_event);
  return FA_OK;
}

FA_API fa_status fa_cta_order(int npairs, int ntiles, int slots, int* group, int* pair, int* tile,
                              long long capacity) {
  if (npairs <= 0 || ntiles <= 0 || slots <= 0) return FA_ERR_SHAPE;
  if (static_cast<long long>(npairs) * ntiles > 0x7fffffffLL) return FA_ERR_SHAPE;
  const int g = fa::pair_group_size(npairs, ntiles, slots);
  if (group) *group = g;
  const long long ctas = fa::grid_ctas(npairs, ntiles, g);
  const long long n = capacity < ctas ? capacity : ctas;
  for (long long b = 0; b < n; ++b) {
    int pr = 0, t = 0;
    fa::item_of_index(static_cast<uint32_t>(b), g, ntiles, pr, t);  // the kernels' own decode of their block index
    if (tile) tile[b] = t;
    if (pair) pair[b] = pr;
  }
  return FA_OK;
}

FA_API fa_status fa_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  FA_TRY(check_arch());
  uint32_t* err = nullptr;
  FA_TRY(error_word(&err));
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;
  const cudaError_t e = fa::launch_wait_timeout_selftest(err, limit_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("self-test launch", e);
}

FA_API fa_status fa_microbench(int which, int iters, double* result, void* stream) {
  if (!result) return FA_ERR_NULL;
  const bool known = (which >= 0 && which <= 11) || which == 38 || which == 40 || which == 42 || which == 43;
  if (!known || iters <= 0 || iters > (1 << 20)) return FA_ERR_SHAPE;
  FA_TRY(check_arch());
  uint32_t* err = nullptr;
  FA_TRY(error_word(&err));
  const cudaError_t e = fa::run_microbench(which, iters, err, result, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("microbenchmark", e);
}

}  // extern "C"
