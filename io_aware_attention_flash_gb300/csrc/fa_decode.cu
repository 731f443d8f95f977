// Split-KV decode forward for sm_103a ("LLM Systems 22: Flash Attention",
// sections 5.1 and 5.2): a few new query tokens per head (Nq <= 8) attend to
// a long key/value cache.  With so few query rows there is one tiny GEMV per
// head, far too little parallel work along the query dimension, and the cost
// is reading K and V once: the work is split along the key/value length, each
// split keeps its own softmax statistics (m, l) and unnormalised output, and a
// light merge combines them.
//
//   fa_decode_split_kernel  persistent (one CTA per SM); CTA c takes work items
//                           c, c + G, ... where item = (sequence·head, split).
//                           The last warp streams the 128-key K and V tiles of
//                           its items through a 3-stage TMA ring without
//                           draining between items; compute warp w owns keys
//                           32·(w mod 4) .. +31 of every tile and a group of
//                           the queries (with two or more queries, two groups:
//                           two warps per SM sub-partition share the keys) and
//                           keeps its own partial softmax (the compute warps
//                           do not synchronise within an item); at the end of
//                           an item the four key quarters' partials are
//                           combined in shared memory into one partial
//                           (m, l, O) per item and query.
//   fa_decode_merge_kernel  one warp per (sequence, head, query): combines the
//                           S partials into O (bf16) and LSE.
//
// The bytes are the cost (K and V once, 4·d bytes per cached token and head),
// so the arithmetic runs on the FMA pipe: lanes split the head dimension for
// q·k, and one 31-shuffle transpose-reduction per query leaves each lane the
// score of one key.  Scores are kept in base-2 units (c = scale·log2 e).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_kernels.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

template <int D, int QG>
struct DecCfg {
  static constexpr int KB = D / 64;                    // 128-byte swizzle blocks per row
  static constexpr int BLK_BYTES = kTile * 128;        // 128 rows x 64 bf16
  static constexpr int TILE_BYTES = KB * BLK_BYTES;    // 128 keys x D
  static constexpr int NST = 3;                        // ring stages (K and V tile each)
  static constexpr int NQMAX = 8;
  static constexpr int E = D / 32;                     // head-dimension elements per lane
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int NCW = 4 * QG;                   // compute warps: 4 key quarters x QG query groups
  static constexpr int OFF_P = OFF_V + NST * TILE_BYTES;  // [NCW][NQMAX][32] fp32 probabilities
  // [QG][4 key quarters][NQMAX / QG queries][D + 2] fp32: each warp's (O, m, l)
  // of an item, combined into one partial per query group by its first warp.
  static constexpr int CMB_STRIDE = D + 2;
  static constexpr int OFF_CMB = OFF_P + NCW * NQMAX * 32 * 4;
  static constexpr int OFF_BAR = OFF_CMB + 4 * NQMAX * CMB_STRIDE * 4;
  static constexpr int B_FULL = 0;
  static constexpr int B_EMPTY = NST;
  static constexpr int B_CFULL = 2 * NST;        // [QG]: a group's four partials are in shared memory
  static constexpr int B_CFREE = 2 * NST + QG;   // [QG]: the group's first warp has read them
  static constexpr int NBAR = 2 * NST + 2 * QG;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // abort flag
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
  static constexpr int NUM_THREADS = 32 * (NCW + 1);   // compute warps, then the TMA warp
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Byte offset, inside a 128-byte swizzled tile, of row j's head-dimension
// elements E·lane .. E·lane + E - 1 (contiguous: 8 bytes for d = 128, 4 for 64).
template <int D>
__device__ __forceinline__ uint32_t row_slice(int j, int lane) {
  constexpr int E = D / 32;
  const int c0 = E * lane;                  // first column
  const int blk = c0 / 64;                  // 64-column block
  const int byte = (c0 % 64) * 2;           // byte inside the 128-byte row of the block
  return blk * (kTile * 128) + j * 128 + ((((byte >> 4) ^ (j & 7)) << 4) | (byte & 15));
}

template <int D>
__device__ __forceinline__ void load_row_slice(uint32_t addr, float (&x)[D / 32]) {
  if constexpr (D == 128) {
    uint32_t a, b;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
    x[0] = bf16lo_to_f32(a);
    x[1] = bf16hi_to_f32(a);
    x[2] = bf16lo_to_f32(b);
    x[3] = bf16hi_to_f32(b);
  } else {
    uint32_t a;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a) : "r"(addr));
    x[0] = bf16lo_to_f32(a);
    x[1] = bf16hi_to_f32(a);
  }
}

// v[i] holds this lane's contribution to element i (32 elements); afterwards
// v[0] holds the sum over all 32 lanes of element `lane`.
__device__ __forceinline__ void transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
}

template <int D, int NQ, int QG>
__global__ void __launch_bounds__(DecCfg<D, QG>::NUM_THREADS, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const DecodeParams p) {
  using C = DecCfg<D, QG>;
  static_assert(NQ % QG == 0, "queries split evenly over the query groups");
  grid_launch_dependents();  // the merge may be scheduled; it waits for this grid to finish
  constexpr int NQW = NQ / QG;  // queries per compute warp
  constexpr int E = C::E;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_base + pad;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = p.B * p.H * p.splits;

  if (warp == C::NCW && lane == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_EMPTY + s), C::NCW * 32);
    }
    for (int g = 0; g < QG; ++g) {
      mbar_init(bar(C::B_CFULL + g), 4 * 32);
      mbar_init(bar(C::B_CFREE + g), 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int t = 0;  // tiles issued by this CTA
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int bh = item / p.splits, split = item - (item / p.splits) * p.splits;
        const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
        const int k_lo = split * p.split_len, k_hi = min(p.Nk, k_lo + p.split_len);
        for (int kt = k_lo; kt < k_hi; kt += kTile, ++t) {
          const int st = t % C::NST;
          if (t >= C::NST && !wait_bounded(bar(C::B_EMPTY + st), ((t / C::NST) - 1) & 1, abort_flag, p.err,
                                           p.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_FULL + st), 2 * C::TILE_BYTES);
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_4d(sb + C::OFF_K + st * C::TILE_BYTES + kb * C::BLK_BYTES, &tmK, bar(C::B_FULL + st),
                        kb * 64, h, kt, b);
            tma_load_4d(sb + C::OFF_V + st * C::TILE_BYTES + kb * C::BLK_BYTES, &tmV, bar(C::B_FULL + st),
                        kb * 64, h, kt, b);
          }
        }
      }
      // Every copy this thread issued lands before it exits, whoever aborted
      // and whenever: this kernel has no CTA-wide barrier at its end, so once
      // the compute warps have left (finished, or aborted after this loop
      // issued its last tile) the CTA would retire with copies still writing
      // into its shared memory.  On a clean run these phases have completed.
      for (int s = 0; s < C::NST && s < t; ++s) {
        const int last = s + ((t - 1 - s) / C::NST) * C::NST;  // last tile issued into stage s
        wait_drain(bar(C::B_FULL + s), (last / C::NST) & 1, p.err, p.timeout_ns);
      }
    }
  } else {
    // ---------------------------------------------------------------- scores, softmax, P·V
    const float c = p.scale_log2;
    const int kw = warp % 4;          // key quarter of every tile
    const int qg = warp / 4;          // query group
    const int q0 = qg * NQW;          // first query of this warp's group
    float* cmb = reinterpret_cast<float*>(smem + C::OFF_CMB) + qg * 4 * NQW * C::CMB_STRIDE;
    int n_done = 0;                   // items this warp has finished
    float* pbuf = reinterpret_cast<float*>(smem + C::OFF_P) + warp * C::NQMAX * 32;
    int t = 0;  // tiles consumed
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int bh = item / p.splits, split = item - (item / p.splits) * p.splits;
      const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
      const int k_lo = split * p.split_len, k_hi = min(p.Nk, k_lo + p.split_len);
      float qv[NQW][E], o[NQW][E], m[NQW], lp[NQW];
#pragma unroll
      for (int qq = 0; qq < NQW; ++qq) {
        const int qi = q0 + qq < p.Nq ? q0 + qq : 0;
        const uint16_t* qrow = p.q + ((static_cast<size_t>(b) * p.Nq + qi) * p.H + h) * D + E * lane;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          qv[qq][e] = __uint_as_float(static_cast<uint32_t>(qrow[e]) << 16);
          o[qq][e] = 0.f;
        }
        m[qq] = -CUDART_INF_F;
        lp[qq] = 0.f;
      }
      for (int kt = k_lo; kt < k_hi; kt += kTile, ++t) {
        const int st = t % C::NST;
        if (!wait_bounded(bar(C::B_FULL + st), (t / C::NST) & 1, abort_flag, p.err, p.timeout_ns)) {
          ok = false;
          break;
        }
        const uint32_t ktile = sb + C::OFF_K + st * C::TILE_BYTES;
        const uint32_t vtile = sb + C::OFF_V + st * C::TILE_BYTES;
        const int key = kt + kw * 32 + lane;  // this lane's key after the reduction
        // ---- scores of this warp's 32 keys, one query at a time (not unrolled:
        // one set of 32 partial dot products live at a time)
        float sc[NQW];
#pragma unroll 1
        for (int qq = 0; qq < NQW; ++qq) {
          float qcur[E];
#pragma unroll
          for (int e = 0; e < E; ++e) qcur[e] = qv[qq][e];
          float part[32];
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            float kx[E];
            load_row_slice<D>(ktile + row_slice<D>(kw * 32 + kk, lane), kx);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc = fmaf(qcur[e], kx[e], acc);
            part[kk] = acc;
          }
          transpose_reduce32(part, lane);
          // Causal: the new tokens are the last Nq positions, so query qq sees
          // keys up to Nk - Nq + qq.
          const int lim = p.causal ? p.Nk - p.Nq + q0 + qq : p.Nk - 1;
          sc[qq] = (q0 + qq < p.Nq && key <= lim && key < p.Nk) ? part[0] * c : -CUDART_INF_F;
        }
        // ---- online softmax over the warp's keys, per query
#pragma unroll
        for (int qq = 0; qq < NQW; ++qq) {
          float mt = sc[qq];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
          const float m_new = fmaxf(m[qq], mt);
          const float alpha = (m[qq] == -CUDART_INF_F) ? 0.f : ex2_approx(m[qq] - m_new);
          const float pr = (sc[qq] == -CUDART_INF_F) ? 0.f : ex2_approx(sc[qq] - m_new);
          lp[qq] = lp[qq] * alpha + pr;
#pragma unroll
          for (int e = 0; e < E; ++e) o[qq][e] *= alpha;
          m[qq] = m_new;
          pbuf[qq * 32 + lane] = pr;
        }
        __syncwarp();
        // ---- O += P V over the warp's 32 keys (lane = head-dimension slice)
#pragma unroll 4
        for (int kk = 0; kk < 32; ++kk) {
          float vx[E];
          load_row_slice<D>(vtile + row_slice<D>(kw * 32 + kk, lane), vx);
#pragma unroll
          for (int qq = 0; qq < NQW; ++qq) {
            const float pq = pbuf[qq * 32 + kk];
#pragma unroll
            for (int e = 0; e < E; ++e) o[qq][e] = fmaf(pq, vx[e], o[qq][e]);
          }
        }
        __syncwarp();
        mbar_arrive(bar(C::B_EMPTY + st));
      }
      if (!ok) break;
      // ---- the item's partial (m, l, unnormalised O) per query: the four key
      // quarters' partials meet in shared memory and the group's first warp
      // combines them (bounded mbarrier waits, so an abort cannot strand a warp).
      if (kw != 0 && n_done > 0 &&
          !wait_bounded(bar(C::B_CFREE + qg), (n_done - 1) & 1, abort_flag, p.err, p.timeout_ns))
        break;
#pragma unroll
      for (int qq = 0; qq < NQW; ++qq) {
        float l = lp[qq];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        float* row = cmb + (kw * NQW + qq) * C::CMB_STRIDE;
#pragma unroll
        for (int e = 0; e < E; ++e) row[E * lane + e] = o[qq][e];
        if (lane == 0) {
          row[D] = m[qq];
          row[D + 1] = l;
        }
      }
      mbar_arrive(bar(C::B_CFULL + qg));
      if (kw == 0) {
        if (!wait_bounded(bar(C::B_CFULL + qg), n_done & 1, abort_flag, p.err, p.timeout_ns)) break;
#pragma unroll
        for (int qq = 0; qq < NQW; ++qq) {
          if (q0 + qq >= p.Nq) break;
          float mk[4], mx = -CUDART_INF_F;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mk[k] = cmb[(k * NQW + qq) * C::CMB_STRIDE + D];
            mx = fmaxf(mx, mk[k]);
          }
          float acc[E], l = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (mk[k] == -CUDART_INF_F) continue;
            const float* row = cmb + (k * NQW + qq) * C::CMB_STRIDE;
            const float w = ex2_approx(mk[k] - mx);
            l = fmaf(w, row[D + 1], l);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(w, row[E * lane + e], acc[e]);
          }
          const size_t idx = static_cast<size_t>(item) * p.Nq + q0 + qq;
          float* op = p.o_part + idx * D + E * lane;
#pragma unroll
          for (int e = 0; e < E; ++e) op[e] = acc[e];
          if (lane == 0) {
            p.ml_part[idx * 2 + 0] = mx;
            p.ml_part[idx * 2 + 1] = l;
          }
        }
        __syncwarp();
        mbar_arrive(bar(C::B_CFREE + qg));
      }
      ++n_done;
    }
  }
}

// ----------------------------------------------------------------------------
// Several new tokens (d = 128): the two products of each 128-key tile on the
// tensor core, with the keys as the M dimension and the queries as N = 16
// (rows past Nq are zero):
//   Sᵀ = K · Qᵀ      A = K tile (K-major), B = Q (16 x d, K-major)  -> TMEM, 16 cols
//   Oᵀ_tile = Vᵀ · Pᵀ  A = V tile read MN-major, B = P (16 x 128 keys, K-major)
// Thread t of warps 0-3 owns TMEM lane t: key t of the tile for Sᵀ and P,
// head dimension t for Oᵀ.  The online softmax runs per query across the four
// warps (tile maxima exchanged through shared memory behind a bounded
// mbarrier); each thread keeps its key's partial row sums and its dimension's
// running output in registers, so the tensor memory holds only per-tile
// results (Sᵀ and Oᵀ_tile, double-buffered: 64 columns).  Warp 4 streams
// K and V through the same 3-stage TMA ring as the FMA kernel; warp 5 issues
// the MMAs.  One partial (m, l, O) per item and query, merged as above.
// ----------------------------------------------------------------------------
struct DecMmaCfg {
  static constexpr int D = 128;
  static constexpr int NQP = 16;                        // queries padded to the MMA's N
  static constexpr int BLK_BYTES = kTile * 128;         // 128 rows x 64 bf16
  static constexpr int TILE_BYTES = 2 * BLK_BYTES;      // 128 keys x 128
  static constexpr int QBLK = NQP * 128;                // 16 rows x 64 bf16
  static constexpr int NST = 3;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + NST * TILE_BYTES;  // Q, 16 x 128, two 64-column blocks
  static constexpr int OFF_P = OFF_Q + 2 * QBLK;          // P[2 buffers], 16 x 128 keys each
  static constexpr int OFF_XCH = OFF_P + 2 * 2 * QBLK;    // [2][4 warps][16] fp32
  static constexpr int OFF_BAR = OFF_XCH + 2 * 4 * NQP * 4;
  static constexpr int B_FULL = 0, B_EMPTY = NST, B_SFULL = 2 * NST, B_PFULL = B_SFULL + 2,
                       B_PVDONE = B_PFULL + 2, B_XCH = B_PVDONE + 2, B_QREADY = B_XCH + 1, B_DRAIN = B_QREADY + 1,
                       NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;     // tmem slot, abort flag
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;
  static constexpr int NUM_THREADS = 6 * 32;
  static constexpr uint32_t TMEM_COLS = 64;               // Sᵀ[2] at 0, 16; Oᵀ_tile[2] at 32, 48
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int NQ>
__global__ void __launch_bounds__(DecMmaCfg::NUM_THREADS, 1)
    fa_decode_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const DecodeParams p) {
  using C = DecMmaCfg;
  constexpr int D = C::D;
  grid_launch_dependents();  // the merge may be scheduled; it waits for this grid to finish
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_base + pad;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = p.B * p.H * p.splits;

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_SFULL + b), 1);
      mbar_init(bar(C::B_PFULL + b), 128);
      mbar_init(bar(C::B_PVDONE + b), 1);
    }
    mbar_init(bar(C::B_XCH), 128);
    mbar_init(bar(C::B_QREADY), 128);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp < 4) {  // P rows past Nq stay zero for good (finite B operand)
    for (int i = threadIdx.x; i < 2 * 2 * C::QBLK / 16; i += 128)
      reinterpret_cast<uint4*>(smem + C::OFF_P)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int t = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int bh = item / p.splits, split = item - (item / p.splits) * p.splits;
        const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
        const int k_lo = split * p.split_len, k_hi = min(p.Nk, k_lo + p.split_len);
        for (int kt = k_lo; kt < k_hi; kt += kTile, ++t) {
          const int st = t % C::NST;
          if (t >= C::NST && !wait_bounded(bar(C::B_EMPTY + st), ((t / C::NST) - 1) & 1, abort_flag, p.err,
                                           p.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_FULL + st), 2 * C::TILE_BYTES);
          for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sb + C::OFF_K + st * C::TILE_BYTES + kb * C::BLK_BYTES, &tmK, bar(C::B_FULL + st),
                        kb * 64, h, kt, b);
            tma_load_4d(sb + C::OFF_V + st * C::TILE_BYTES + kb * C::BLK_BYTES, &tmV, bar(C::B_FULL + st),
                        kb * 64, h, kt, b);
          }
        }
      }
      // As in the FMA kernel: every issued copy lands before the CTA-wide
      // barrier at the end, whoever aborted and whenever.
      for (int s = 0; s < C::NST && s < t; ++s) {
        const int last = s + ((t - 1 - s) / C::NST) * C::NST;
        wait_drain(bar(C::B_FULL + s), (last / C::NST) & 1, p.err, p.timeout_ns);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, C::NQP, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(D, C::NQP, true, false);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 16, 1024);          // K tile, K-major
      const uint64_t dV0 = sdesc_sw128(sb + C::OFF_V, C::BLK_BYTES, 1024);  // V tile as the MN-major A of Vᵀ
      const uint64_t dQ = sdesc_sw128(sb + C::OFF_Q, 16, 1024);
      const uint64_t dP0 = sdesc_sw128(sb + C::OFF_P, 16, 1024);
      // Sᵀ of tile u (K from ring slot u mod 3, into TMEM buffer u mod 2).
      auto issue_s = [&](int u) -> bool {
        const int st = u % C::NST, bf = u & 1;
        if (!wait_bounded(bar(C::B_FULL + st), (u / C::NST) & 1, abort_flag, p.err, p.timeout_ns)) return false;
        tc_fence_after();
        const uint64_t dK = sdesc_add(dK0, st * C::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk / 4) * C::BLK_BYTES + (kk % 4) * 32, qoff = (kk / 4) * C::QBLK + (kk % 4) * 32;
          mma_ss(tmem + 16 * bf, sdesc_add(dK, koff), sdesc_add(dQ, qoff), idesc_s, kk > 0);
        }
        tc_commit(bar(C::B_SFULL + bf));
        return true;
      };
      int t = 0, n_item = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++n_item) {
        const int split = item - (item / p.splits) * p.splits;
        const int k_lo = split * p.split_len, k_hi = min(p.Nk, k_lo + p.split_len);
        if (!wait_bounded(bar(C::B_QREADY), n_item & 1, abort_flag, p.err, p.timeout_ns)) break;
        // Within an item Sᵀ of the next tile is issued before this tile's P is
        // awaited (its TMEM buffer was read before the previous P arrived);
        // across items it cannot be, as the next item's Q is staged only
        // after this item's last output has been taken.
        if (!issue_s(t)) break;
        for (int kt = k_lo; kt < k_hi; kt += kTile, ++t) {
          const int st = t % C::NST, bf = t & 1;
          if (kt + kTile < k_hi && !issue_s(t + 1)) {
            ok = false;
            break;
          }
          if (!wait_bounded(bar(C::B_PFULL + bf), (t >> 1) & 1, abort_flag, p.err, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dV = sdesc_add(dV0, st * C::TILE_BYTES), dP = sdesc_add(dP0, bf * 2 * C::QBLK);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ss(tmem + 32 + 16 * bf, sdesc_add(dV, kk * 2048), sdesc_add(dP, (kk / 4) * C::QBLK + (kk % 4) * 32),
                   idesc_o, kk > 0);
          tc_commit(bar(C::B_PVDONE + bf));
          tc_commit(bar(C::B_EMPTY + st));
        }
      }
      tc_commit(bar(C::B_DRAIN));
      wait_drain(bar(C::B_DRAIN), 0, p.err, p.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------------- softmax, P, running O
    const float c = p.scale_log2;
    const int r = warp * 32 + lane;  // TMEM lane: key of the tile (Sᵀ, P), head dimension (Oᵀ)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
    int t = 0, nx = 0, n_item = 0;
    bool ok = true;
    // One exchange of a value per query among the four warps: warp maxima or
    // sums in, the four per query out (mbarrier with a bounded wait).
    auto exchange = [&](float (&v)[NQ], float (&out)[4][NQ]) -> bool {
      float* slot = xch + (nx & 1) * 4 * C::NQP;
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (lane == q) slot[warp * C::NQP + q] = v[q];
      mbar_arrive(bar(C::B_XCH));
      const bool got = wait_bounded(bar(C::B_XCH), nx & 1, abort_flag, p.err, p.timeout_ns);
      ++nx;
      if (!got) return false;
#pragma unroll
      for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int q = 0; q < NQ; ++q) out[w][q] = slot[w * C::NQP + q];
      return true;
    };
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++n_item) {
      const int bh = item / p.splits, split = item - (item / p.splits) * p.splits;
      const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
      const int k_lo = split * p.split_len, k_hi = min(p.Nk, k_lo + p.split_len);
      // Q of this item into the 128-byte swizzled B layout (rows past Nq zero);
      // every MMA that read the previous item's Q has completed (its Sᵀ was waited for).
      for (int i = r; i < C::NQP * 16; i += 128) {
        const int row = i / 16, c16 = i % 16;  // 16-byte chunk along d
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < p.Nq)
          v = *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(b) * p.Nq + row) * p.H + h) * D + c16 * 8);
        *reinterpret_cast<uint4*>(smem + C::OFF_Q + (c16 / 8) * C::QBLK + row * 128 + (((c16 % 8) ^ (row & 7)) * 16)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_QREADY));
      float m[NQ], lsum[NQ], ov[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        m[q] = -CUDART_INF_F;
        lsum[q] = 0.f;
        ov[q] = 0.f;
      }
      for (int kt = k_lo; kt < k_hi; kt += kTile, ++t) {
        const int bf = t & 1;
        if (!wait_bounded(bar(C::B_SFULL + bf), (t >> 1) & 1, abort_flag, p.err, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16(lane_addr + 16 * bf, sv);
        tmem_wait_ld();
        reg_fence(sv);
        const int key = kt + r;
        float x[NQ], wm[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const int lim = p.causal ? p.Nk - p.Nq + q : p.Nk - 1;  // last key query q sees
          x[q] = (q < p.Nq && key <= lim && key < p.Nk) ? __uint_as_float(sv[q]) * c : -CUDART_INF_F;
          wm[q] = x[q];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) wm[q] = fmaxf(wm[q], __shfl_xor_sync(0xffffffffu, wm[q], off));
        }
        float all[4][NQ];
        if (!exchange(wm, all)) {
          ok = false;
          break;
        }
        float alpha[NQ];
        const uint32_t prow = C::OFF_P + bf * 2 * C::QBLK + (r / 64) * C::QBLK;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const float m_new = fmaxf(fmaxf(m[q], fmaxf(all[0][q], all[1][q])), fmaxf(all[2][q], all[3][q]));
          alpha[q] = (m[q] == -CUDART_INF_F) ? 0.f : ex2_approx(m[q] - m_new);
          const float pq = (x[q] == -CUDART_INF_F) ? 0.f : ex2_approx(x[q] - m_new);
          lsum[q] = fmaf(lsum[q], alpha[q], pq);
          m[q] = m_new;
          // P[q][key r]: row q of the K-major B operand, keys contiguous
          const uint32_t byte = (r % 64) * 2;
          const uint16_t pb = static_cast<uint16_t>(pack_bf16x2(pq, 0.f));
          *reinterpret_cast<uint16_t*>(smem + prow + q * 128 + ((((byte >> 4) ^ (q & 7)) << 4) | (byte & 15))) = pb;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_PFULL + bf));
        if (!wait_bounded(bar(C::B_PVDONE + bf), (t >> 1) & 1, abort_flag, p.err, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t ot[16];
        tmem_ld16(lane_addr + 32 + 16 * bf, ot);
        tmem_wait_ld();
        reg_fence(ot);
#pragma unroll
        for (int q = 0; q < NQ; ++q) ov[q] = fmaf(ov[q], alpha[q], __uint_as_float(ot[q]));
      }
      if (!ok) break;
      // ---- the item's partial per query: l summed over the 128 keys' threads
      float ws[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        ws[q] = lsum[q];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ws[q] += __shfl_xor_sync(0xffffffffu, ws[q], off);
      }
      float all[4][NQ];
      if (!exchange(ws, all)) break;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q >= p.Nq) break;
        const size_t idx = static_cast<size_t>(item) * p.Nq + q;
        p.o_part[idx * D + r] = ov[q];
        if (r == 0) {
          p.ml_part[idx * 2 + 0] = m[q];
          p.ml_part[idx * 2 + 1] = (all[0][q] + all[1][q]) + (all[2][q] + all[3][q]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// One warp per (sequence, head, query): O = Σ 2^(m_p − m) O_p / Σ 2^(m_p − m) l_p
// over the splits partials of the head, m = max m_p; LSE = ln 2 · (m + log2 l).
// The partials' weights are formed 32 at a time, one per lane, and the O
// partials are then read with several loads in flight (no load waits on
// another).
template <int D>
__global__ void __launch_bounds__(64) fa_decode_merge_kernel(const DecodeParams p) {
  constexpr int E = D / 32;
  grid_dependency_wait();  // the partials of the split kernel are complete
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= p.B * p.H * p.Nq) return;
  const int qq = wid % p.Nq, bh = wid / p.Nq;
  const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
  const int n_part = p.splits;
  const size_t part0 = static_cast<size_t>(bh) * n_part;
  float mmax = -CUDART_INF_F;
  for (int i = lane; i < n_part; i += 32) mmax = fmaxf(mmax, p.ml_part[((part0 + i) * p.Nq + qq) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, off));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float l = 0.f;
  if (mmax != -CUDART_INF_F) {
    for (int i0 = 0; i0 < n_part; i0 += 32) {
      float w = 0.f;  // this lane's partial: i0 + lane
      if (i0 + lane < n_part) {
        const size_t idx = (part0 + i0 + lane) * p.Nq + qq;
        const float mp = p.ml_part[idx * 2];
        if (mp != -CUDART_INF_F) {
          w = ex2_approx(mp - mmax);
          l = fmaf(w, p.ml_part[idx * 2 + 1], l);
        }
      }
      const int cnt = min(32, n_part - i0);
#pragma unroll 8
      for (int j = 0; j < cnt; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, j);
        const float* op = p.o_part + ((part0 + i0 + j) * p.Nq + qq) * D + E * lane;
        float v[E];
        if constexpr (E == 4) {
          const float4 t = *reinterpret_cast<const float4*>(op);
          v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(op);
          v[0] = t.x, v[1] = t.y;
        }
        if (wj != 0.f) {
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(wj, v[e], acc[e]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  }
  const float inv_l = l > 0.f ? 1.0f / l : 0.f;
  uint16_t* orow = p.o + ((static_cast<size_t>(b) * p.Nq + qq) * p.H + h) * D + E * lane;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t*>(orow + e) = pack_bf16x2(acc[e] * inv_l, acc[e + 1] * inv_l);
  if (lane == 0)
    p.lse[(static_cast<size_t>(b) * p.H + h) * p.Nq + qq] = l > 0.f ? (mmax + log2f(l)) * kLn2 : -CUDART_INF_F;
}

template <int D, int NQ>
cudaError_t launch_decode_dq(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                             cudaStream_t s) {
  constexpr int QG = NQ >= 2 ? 2 : 1;
  using C = DecCfg<D, QG>;
  static SmemLimit smem_limit;
  cudaError_t e =
      smem_limit.ensure(reinterpret_cast<const void*>(fa_decode_split_kernel<D, NQ, QG>), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  fa_decode_split_kernel<D, NQ, QG><<<grid, C::NUM_THREADS, C::SMEM_BYTES, s>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = static_cast<long long>(p.B) * p.H * p.Nq;
  // Two warps per block: the rows are few (B·H·Nq), so spread them over the SMs.
  // The merge is scheduled while the split kernel's last items run and
  // waits for it before reading the partials.
  return launch_kernel(fa_decode_merge_kernel<D>, dim3(static_cast<unsigned>((warps * 32 + 63) / 64)), dim3(64), 0, s,
                       true, p);
}

template <int NQ>
cudaError_t launch_decode_mma(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                              cudaStream_t s) {
  using C = DecMmaCfg;
  static SmemLimit smem_limit;
  cudaError_t e = smem_limit.ensure(reinterpret_cast<const void*>(fa_decode_mma_kernel<NQ>), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  fa_decode_mma_kernel<NQ><<<grid, C::NUM_THREADS, C::SMEM_BYTES, s>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = static_cast<long long>(p.B) * p.H * p.Nq;
  return launch_kernel(fa_decode_merge_kernel<C::D>, dim3(static_cast<unsigned>((warps * 32 + 63) / 64)), dim3(64), 0,
                       s, true, p);
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                            cudaStream_t s) {
  if (D == 128 && p.Nq >= 2) {  // several new tokens: the tensor-core kernel
    if (p.Nq <= 2) return launch_decode_mma<2>(tk, tv, p, grid, s);
    if (p.Nq <= 4) return launch_decode_mma<4>(tk, tv, p, grid, s);
    return launch_decode_mma<8>(tk, tv, p, grid, s);
  }
  if (p.Nq <= 1) return launch_decode_dq<D, 1>(tk, tv, p, grid, s);
  if (p.Nq <= 2) return launch_decode_dq<D, 2>(tk, tv, p, grid, s);
  if (p.Nq <= 4) return launch_decode_dq<D, 4>(tk, tv, p, grid, s);
  return launch_decode_dq<D, 8>(tk, tv, p, grid, s);
}

}  // namespace

cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                          cudaStream_t s) {
  if (d == 64) return launch_decode_d<64>(tk, tv, p, grid, s);
  return launch_decode_d<128>(tk, tv, p, grid, s);
}

}  // namespace fa
