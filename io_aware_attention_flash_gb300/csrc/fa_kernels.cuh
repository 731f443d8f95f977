// Parameters and launch entry points shared between the C ABI layer and the
// kernels.  Internal to libfa_gb300.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr int kTile = 128;           // query rows per Q tile and keys per K/V tile
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

// Where a CTA's rows live.  Dense batches: sequence b is rows b*N .. b*N+N-1
// of the [B*N, H, d] view and TMA coordinates use (row, b) with the batch as
// the outer tensor dimension, so reads past N zero-fill.  Packed batches:
// sequence s is rows cu[s] .. cu[s+1]-1 of the single [total, H, d] tensor.
struct SeqView {
  const int* cu_seqlens;  // device [nseq + 1] or nullptr for a dense batch
  int H;
  int N;                  // dense: rows per sequence; packed: total rows
  int lse_stride;         // N (dense) or max_seqlen (packed)
  int npairs;             // (sequence, head) pairs: nseq·H
  int ntiles;             // tiles of the launch's kind along the longest sequence
  int pair_group;         // pairs per launch group (pair_group_size)
};

// CTA order.  A CTA's work item is a (sequence·head pair, tile), and CTAs
// start in increasing linear block index.  The items are launched in groups
// of consecutive pairs: every tile of a group, tile-major in the kernel's
// heaviest-first tile order, then the next group.  The CTAs in flight then
// share the tiles of a few pairs in L2 (a packed batch with hundreds of
// pairs would otherwise have nearly every CTA in flight on a pair of its
// own, and at long sequences the K/V or Q/dO/dQ rows of all pairs would not
// fit in L2).  A freed SM takes the next CTA, so starting each group's heavy
// tiles first keeps the causal load balance as long as the groups are equal
// and each spans at least one wave of CTAs; a shorter group, or a last group
// smaller than the others, leaves heavy tiles for the end (greedy schedules
// of the causal tile costs: 20-30 % longer).  Group size: the smallest
// divisor of the pair count with at least one wave of tiles (searched up to
// 4x that size); all pairs (plain tile-major order) when there is none.
inline int pair_group_size(int npairs, int ntiles, int slots) {
  const long long need = (static_cast<long long>(slots) + ntiles - 1) / ntiles;
  for (long long g = need; g < npairs && g <= 4 * need; ++g)
    if (npairs % g == 0) return static_cast<int>(g);
  return npairs;
}

// Multiprocessors of the current device (cached per host thread).
inline cudaError_t current_sm_count(int& sms) {
  thread_local int cached_dev = -1, cached_sms = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev != cached_dev) {
    e = cudaDeviceGetAttribute(&cached_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cached_dev = dev;
  }
  sms = cached_sms;
  return cudaSuccess;
}

inline long long grid_ctas(int npairs, int ntiles, int group) {
  return static_cast<long long>((npairs + group - 1) / group) * group * ntiles;
}

// Work item (pair, tile) of linear launch index b under groups of `group`
// pairs of `ntiles` tiles each; pair >= npairs marks an index of the last,
// partial group with no work.  The kernels decode their work items with it
// and fa_cta_order reports the launch order with it on the host.  Launches
// are limited to 2^31 - 1 items, so 32-bit unsigned arithmetic suffices (a
// 64-bit division would cost the kernels' lean warps registers).
__host__ __device__ __forceinline__ void item_of_index(uint32_t b, uint32_t group, uint32_t ntiles, int& pair,
                                                       int& tile) {
  const uint32_t per_group = group * ntiles;
  const uint32_t grp = b / per_group;
  const uint32_t r = b - grp * per_group;
  const uint32_t t = r / group;
  tile = static_cast<int>(t);
  pair = static_cast<int>(grp * group + (r - t * group));
}

// (pair, tile) of this CTA.
__device__ __forceinline__ void cta_item(const SeqView& sv, int& pair, int& tile) {
  item_of_index(blockIdx.x, sv.pair_group, sv.ntiles, pair, tile);
}

constexpr int kMaxDevices = 64;

// Raises a kernel's dynamic shared-memory limit above the 48 KB default.  The
// attribute belongs to the current device, so it is set once per device (and
// per kernel: one object per kernel instantiation), safely across host
// threads.
class SmemLimit {
 public:
  cudaError_t ensure(const void* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (!done_[dev]) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e != cudaSuccess) return e;
      done_[dev] = true;
    }
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

struct FwdParams {
  SeqView sv;
  uint16_t* o;            // bf16 [.., H, d]
  float* lse;             // fp32 [nseq|B, H, lse_stride]
  float scale_log2;       // scale * log2(e)
  int causal;
  uint32_t* err;          // device error word
  uint64_t timeout_ns;
};

struct BwdParams {
  SeqView sv;
  const uint16_t* o;
  const uint16_t* dout;
  const float* lse;
  float* dpsum;           // D = rowsum(dO * O), fp32 [nseq|B, H, lse_stride]
  float* dq_accum;        // fp32, same layout as q ([rows, H, d])
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  float scale;
  float scale_log2;
  int causal;
  int rows;               // B*N (dense) or total (packed): rows of the [rows, H, d] view
  int nseq;               // B (dense) or nseq (packed)
  uint32_t* err;
  uint64_t timeout_ns;
};

// Split-KV decode (fa_decode.cu): q [B, Nq, H, d] against k, v [B, Nk, H, d].
struct DecodeParams {
  const uint16_t* q;      // bf16 [B, Nq, H, d]
  uint16_t* o;            // bf16 [B, Nq, H, d]
  float* lse;             // fp32 [B, H, Nq]
  float* o_part;          // fp32 [B·H·splits, Nq, d]: unnormalised partial outputs
  float* ml_part;         // fp32 [B·H·splits, Nq, 2]: (max, sum) of each partial, base 2
  int B, H, Nq, Nk;
  int splits;             // key/value splits per (sequence, head)
  int split_len;          // keys per split, a multiple of 128
  float scale_log2;
  int causal;             // new tokens are the last Nq positions (lower-right alignment)
  uint32_t* err;
  uint64_t timeout_ns;
};

// Position of a (sequence, head) pair: pair = sequence * H + head.
struct SeqPos {
  int bs, h, seq_start, seqlen, row_base, tma_row0, tma_b;
};

__device__ __forceinline__ SeqPos seq_pos(const SeqView& sv, int pair) {
  SeqPos s;
  s.bs = pair / sv.H;
  s.h = pair % sv.H;
  if (sv.cu_seqlens) {
    s.seq_start = __ldg(sv.cu_seqlens + s.bs);
    s.seqlen = __ldg(sv.cu_seqlens + s.bs + 1) - s.seq_start;
    s.row_base = s.seq_start;
    s.tma_row0 = s.seq_start;
    s.tma_b = 0;
  } else {
    s.seq_start = 0;
    s.seqlen = sv.N;
    s.row_base = s.bs * sv.N;
    s.tma_row0 = 0;
    s.tma_b = s.bs;
  }
  return s;
}

// Launch with or without programmatic stream serialisation (the kernel may
// start before the previous kernel in the stream has finished; it orders its
// dependent reads with grid_dependency_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool overlap_previous, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap_previous ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Grid sizes / launches (defined next to the kernels).
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, int nseq, int max_seqlen, cudaStream_t s);
cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdParams& p, int max_seqlen,
                       cudaStream_t s,
                       cudaEvent_t main_start = nullptr, cudaEvent_t main_end = nullptr);
cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                          cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t run_microbench(int which, int iters, uint32_t* err, double* result, cudaStream_t s);

}  // namespace fa
