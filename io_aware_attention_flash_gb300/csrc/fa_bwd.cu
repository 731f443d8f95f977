// Backward attention kernels for sm_103a.
//
// The backward recomputes the attention tile on chip from Q, K and the saved
// row log-sum-exp instead of reading a stored P ("LLM Systems 22: Flash
// Attention", section 3.2; "08 · FlashAttention", section 三).  Three
// launches:
//   fa_bwd_pre   D_i = Σ_k dO_ik O_ik per row (equal to Σ_j P_ij dP_ij), and
//                zero the fp32 dQ accumulator.
//   fa_bwd_main  one CTA per 128-key tile j of one (sequence, head); loops
//                over the query tiles i that see it (i >= j when causal), the
//                key/value-outer order of the seekfood article's section 1 /
//                3.2 loop, so dK_j and dV_j stay in TMEM for the whole loop:
//                  Sᵀ  = K_j Q_iᵀ              SMEM x SMEM -> TMEM
//                  dPᵀ = V_j dO_iᵀ             SMEM x SMEM -> TMEM
//                  Pᵀ  = 2^(c·Sᵀ − log2e·LSE_i)        (recomputed)
//                  dSᵀ = Pᵀ ∘ (dPᵀ − D_i)
//                  dV_j += Pᵀ dO_i             TMEM(A) x SMEM -> TMEM
//                  dK_j += dSᵀ Q_i             TMEM(A) x SMEM -> TMEM
//                  dQ_i  = dS K_j              SMEM(A, MN-major) x SMEM -> TMEM
//                dQ_i is drained from TMEM by a second warpgroup and added to
//                the fp32 accumulator with vector atomics (other key tiles add
//                to the same rows).
//   fa_bwd_post  dQ = bf16(scale · dQ_accum).
// Warp roles in fa_bwd_main: warps 0-3 recompute P and dS (thread r owns key
// row r = TMEM lane r), warps 4-7 drain dQ and write dV, warp 8 issues TMA,
// warp 9 issues tcgen05.mma.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_kernels.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

// ----------------------------------------------------------------------------
// Row helpers for the [rows, H, d] view
// ----------------------------------------------------------------------------
// Sequence index and row within the sequence of global row g.  Packed
// batches: the largest s in [0, nseq) with cu[s] <= g (binary search; cu is
// non-decreasing, so empty sequences are skipped).
__device__ __forceinline__ void locate_row(const SeqView& sv, int nseq, int g, int& bs, int& local) {
  if (!sv.cu_seqlens) {
    bs = g / sv.N;
    local = g - bs * sv.N;
    return;
  }
  int lo = 0, hi = nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(sv.cu_seqlens + mid) <= g) lo = mid; else hi = mid - 1;
  }
  bs = lo;
  local = g - __ldg(sv.cu_seqlens + lo);
}

// ----------------------------------------------------------------------------
// fa_bwd_pre: one warp per (row, head).
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.sv.H;
  if (wid >= p.rows * H) return;
  const int g = wid / H, h = wid - (wid / H) * H;
  const size_t base = (static_cast<size_t>(g) * H + h) * D;
  constexpr int E = D / 32;  // elements per lane (2 or 4)
  float acc = 0.f;
  if constexpr (E == 4) {
    const uint2 o = *reinterpret_cast<const uint2*>(p.o + base + lane * 4);
    const uint2 d = *reinterpret_cast<const uint2*>(p.dout + base + lane * 4);
    acc = bf16lo_to_f32(o.x) * bf16lo_to_f32(d.x) + bf16hi_to_f32(o.x) * bf16hi_to_f32(d.x) +
          bf16lo_to_f32(o.y) * bf16lo_to_f32(d.y) + bf16hi_to_f32(o.y) * bf16hi_to_f32(d.y);
    *reinterpret_cast<float4*>(p.dq_accum + base + lane * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    const uint32_t o = *reinterpret_cast<const uint32_t*>(p.o + base + lane * 2);
    const uint32_t d = *reinterpret_cast<const uint32_t*>(p.dout + base + lane * 2);
    acc = bf16lo_to_f32(o) * bf16lo_to_f32(d) + bf16hi_to_f32(o) * bf16hi_to_f32(d);
    *reinterpret_cast<float2*>(p.dq_accum + base + lane * 2) = make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    int bs, local;
    locate_row(p.sv, p.nseq, g, bs, local);
    p.dpsum[(static_cast<size_t>(bs) * H + h) * p.sv.lse_stride + local] = acc;
  }
}

// ----------------------------------------------------------------------------
// fa_bwd_post: 8 elements per thread.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const BwdParams p, size_t n8) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(p.dq_accum)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(p.dq_accum)[2 * i + 1];
  const float s = p.scale;
  uint4 w;
  w.x = pack_bf16x2(a.x * s, a.y * s);
  w.y = pack_bf16x2(a.z * s, a.w * s);
  w.z = pack_bf16x2(b.x * s, b.y * s);
  w.w = pack_bf16x2(b.z * s, b.w * s);
  reinterpret_cast<uint4*>(p.dq)[i] = w;
}

// ----------------------------------------------------------------------------
// fa_bwd_main
// ----------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  static constexpr int KB = D / 64;
  static constexpr int BLK_BYTES = kTile * 128;        // 128 rows x 64 bf16
  static constexpr int TILE_BYTES = KB * BLK_BYTES;    // 128 x D bf16
  static constexpr int NSQ = (D == 128) ? 2 : 3;       // Q / dO ring depth
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + NSQ * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + NSQ * TILE_BYTES;      // dSᵀ, 128 key rows x 128 q, 2 blocks
  static constexpr int OFF_STAT = OFF_DS + 2 * BLK_BYTES;       // [2][2][128] fp32: log2e·LSE and D
  static constexpr int OFF_BAR = OFF_STAT + 2 * 2 * kTile * 4;
  static constexpr int B_KV = 0;
  static constexpr int B_QFULL = 1;
  static constexpr int B_DOFULL = B_QFULL + NSQ;
  static constexpr int B_QEMPTY = B_DOFULL + NSQ;
  static constexpr int B_SFULL = B_QEMPTY + NSQ;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_DSREADY = B_DPFULL + 1;
  static constexpr int B_DQFULL = B_DSREADY + 1;
  static constexpr int B_DQDRAINED = B_DQFULL + 1;
  static constexpr int B_DKDV = B_DQDRAINED + 1;
  static constexpr int B_DRAIN = B_DKDV + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // Whatever is left of the 227 KB opt-in limit is alignment slack.
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024 <= 232448) ? SMEM_USED + 1024 : 232448;
  static constexpr int NUM_THREADS = 10 * 32;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t DV_COL = 0;
  static constexpr uint32_t DK_COL = D;
  static constexpr uint32_t S_COL = 2 * D;             // Sᵀ, then Pᵀ (bf16), then dQ_i
  static constexpr uint32_t DP_COL = 2 * D + 128;      // dPᵀ, then dSᵀ (bf16)
  static_assert(SMEM_USED <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::NUM_THREADS, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  if (pad + C::SMEM_USED > C::SMEM_BYTES) {  // uniform across the CTA, before any barrier use
    if (threadIdx.x == 0) atomicOr(p.err, kDevErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_base + pad;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);  // [buf][0: lse2, 1: D][128]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const SeqPos sp = seq_pos(p.sv);
  const int j = blockIdx.y;           // key tile; heavy (small j) tiles first under a causal mask
  const int kv0 = j * kTile;
  if (kv0 >= sp.seqlen) return;
  const int nq_total = (sp.seqlen + kTile - 1) / kTile;
  const int i_first = p.causal ? j : 0;
  const int nq = nq_total - i_first;

  if (warp == C::PRODUCER_WARP && lane == 0) {
    mbar_init(bar(C::B_KV), 1);
    for (int s = 0; s < C::NSQ; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1);
      mbar_init(bar(C::B_DOFULL + s), 1);
      mbar_init(bar(C::B_QEMPTY + s), 1);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_DSREADY), 128);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQDRAINED), 128);
    mbar_init(bar(C::B_DKDV), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const size_t stat_base = (static_cast<size_t>(sp.bs) * p.sv.H + sp.h) * p.sv.lse_stride;
  const size_t row_stride = static_cast<size_t>(p.sv.H) * D;  // elements between consecutive rows

  if (warp == C::PRODUCER_WARP) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILE_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_4d(sb + C::OFF_K + kb * C::BLK_BYTES, &tmK, bar(C::B_KV), kb * 64, sp.h, sp.tma_row0 + kv0,
                    sp.tma_b);
        tma_load_4d(sb + C::OFF_V + kb * C::BLK_BYTES, &tmV, bar(C::B_KV), kb * 64, sp.h, sp.tma_row0 + kv0,
                    sp.tma_b);
      }
      int fills = 0;
      for (int ii = 0; ii < nq; ++ii) {
        const int qs = ii % C::NSQ;
        const int qrow = sp.tma_row0 + (i_first + ii) * kTile;
        if (ii >= C::NSQ && !wait_bounded(bar(C::B_QEMPTY + qs), ((ii / C::NSQ) - 1) & 1, abort_flag, p.err,
                                          p.timeout_ns))
          break;
        mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_4d(sb + C::OFF_Q + qs * C::TILE_BYTES + kb * C::BLK_BYTES, &tmQ, bar(C::B_QFULL + qs),
                      kb * 64, sp.h, qrow, sp.tma_b);
        mbar_arrive_expect_tx(bar(C::B_DOFULL + qs), C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_4d(sb + C::OFF_DO + qs * C::TILE_BYTES + kb * C::BLK_BYTES, &tmdO, bar(C::B_DOFULL + qs),
                      kb * 64, sp.h, qrow, sp.tma_b);
        ++fills;
      }
      if (*abort_flag) {
        wait_drain(bar(C::B_KV), 0, p.err, p.timeout_ns);
        for (int s = 0; s < C::NSQ && s < fills; ++s) {
          const uint32_t ph = ((s + ((fills - 1 - s) / C::NSQ) * C::NSQ) / C::NSQ) & 1;
          wait_drain(bar(C::B_QFULL + s), ph, p.err, p.timeout_ns);
          wait_drain(bar(C::B_DOFULL + s), ph, p.err, p.timeout_ns);
        }
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_sp = idesc_bf16(128, 128, false, false);   // Sᵀ, dPᵀ
      constexpr uint32_t idesc_kv = idesc_bf16(128, D, false, true);      // dV, dK (A from TMEM)
      constexpr uint32_t idesc_q = idesc_bf16(128, D, true, true);        // dQ (A = dS, MN-major)
      const uint32_t tS = tmem + C::S_COL, tDP = tmem + C::DP_COL;
      bool ok = wait_bounded(bar(C::B_KV), 0, abort_flag, p.err, p.timeout_ns);
      for (int ii = 0; ok && ii < nq; ++ii) {
        const int qs = ii % C::NSQ;
        const uint32_t ph = (ii / C::NSQ) & 1;
        const uint32_t sQ = sb + C::OFF_Q + qs * C::TILE_BYTES;
        const uint32_t sdO = sb + C::OFF_DO + qs * C::TILE_BYTES;
        ok = wait_bounded(bar(C::B_QFULL + qs), ph, abort_flag, p.err, p.timeout_ns);
        if (ok && ii > 0) ok = wait_bounded(bar(C::B_DQDRAINED), (ii - 1) & 1, abort_flag, p.err, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk / 4) * C::BLK_BYTES + (kk % 4) * 32;
          mma_ss(tS, sdesc_sw128(sb + C::OFF_K + koff, 16, 1024), sdesc_sw128(sQ + koff, 16, 1024), idesc_sp,
                 kk > 0);
        }
        tc_commit(bar(C::B_SFULL));
        if (!wait_bounded(bar(C::B_DOFULL + qs), ph, abort_flag, p.err, p.timeout_ns)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk / 4) * C::BLK_BYTES + (kk % 4) * 32;
          mma_ss(tDP, sdesc_sw128(sb + C::OFF_V + koff, 16, 1024), sdesc_sw128(sdO + koff, 16, 1024), idesc_sp,
                 kk > 0);
        }
        tc_commit(bar(C::B_DPFULL));
        if (!wait_bounded(bar(C::B_DSREADY), ii & 1, abort_flag, p.err, p.timeout_ns)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t moff = kk * 2048;  // 16 query rows of the MN-major operand
          mma_ts(tmem + C::DV_COL, tS + kk * 8, sdesc_sw128(sdO + moff, C::BLK_BYTES, 1024), idesc_kv,
                 (ii > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::DK_COL, tDP + kk * 8, sdesc_sw128(sQ + moff, C::BLK_BYTES, 1024), idesc_kv,
                 (ii > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(C::B_QEMPTY + qs));
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t moff = kk * 2048;  // 16 key rows
          mma_ss(tS, sdesc_sw128(sb + C::OFF_DS + moff, C::BLK_BYTES, 1024),
                 sdesc_sw128(sb + C::OFF_K + moff, C::BLK_BYTES, 1024), idesc_q, kk > 0);
        }
        tc_commit(bar(C::B_DQFULL));
      }
      if (ok) tc_commit(bar(C::B_DKDV));
      tc_commit(bar(C::B_DRAIN));
      wait_drain(bar(C::B_DRAIN), 0, p.err, p.timeout_ns);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- P, dS
    const int r = warp * 32 + lane;        // key row within the tile = TMEM lane
    const int kv_row = kv0 + r;
    const bool row_dead = kv_row >= sp.seqlen;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t tS = lane_addr + C::S_COL, tDP = lane_addr + C::DP_COL;
    const float c = p.scale_log2;
    const uint32_t sDS = sb + C::OFF_DS;
    bool ok = true;
    for (int ii = 0; ii < nq; ++ii) {
      const int qi = i_first + ii;
      const int q0 = qi * kTile;
      float* lse2 = stat + (ii & 1) * 256;
      float* dsum = lse2 + 128;
      {
        const int q = q0 + r;
        const bool valid = q < sp.seqlen;
        lse2[r] = valid ? __ldg(p.lse + stat_base + q) * kLog2e : CUDART_INF_F;
        dsum[r] = valid ? __ldg(p.dpsum + stat_base + q) : 0.f;
      }
      named_bar_sync(1, 128);
      ok = wait_bounded(bar(C::B_SFULL), ii & 1, abort_flag, p.err, p.timeout_ns) &&
           wait_bounded(bar(C::B_DPFULL), ii & 1, abort_flag, p.err, p.timeout_ns);
      if (ok && ii > 0) ok = wait_bounded(bar(C::B_DQFULL), (ii - 1) & 1, abort_flag, p.err, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = row_dead || (p.causal && qi == j);
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t s[32], dp[32];
        tmem_ld32(tS + ch * 32, s);
        tmem_ld32(tDP + ch * 32, dp);
        tmem_wait_ld();
        reg_fence(s);
        reg_fence(dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = ch * 32 + 2 * e + u;
            float pe = ex2_approx(fmaf(__uint_as_float(s[2 * e + u]), c, -lse2[col]));
            if (need_mask && (row_dead || q0 + col < kv_row)) pe = 0.f;
            pv[u] = pe;
            dv[u] = pe * (__uint_as_float(dp[2 * e + u]) - dsum[col]);
          }
          pk[e] = pack_bf16x2(pv[0], pv[1]);
          dk[e] = pack_bf16x2(dv[0], dv[1]);
        }
        tmem_st16(tS + ch * 16, pk);
        tmem_st16(tDP + ch * 16, dk);
        // dSᵀ row r, query columns ch*32 .. ch*32+31 -> 128-byte swizzled block (ch / 2)
        const uint32_t rowaddr = sDS + (ch >> 1) * C::BLK_BYTES + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t chunk = ((ch & 1) * 4 + u) ^ (r & 7);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowaddr + chunk * 16), "r"(dk[4 * u]),
                       "r"(dk[4 * u + 1]), "r"(dk[4 * u + 2]), "r"(dk[4 * u + 3])
                       : "memory");
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSREADY));
    }
    if (ok) ok = wait_bounded(bar(C::B_DKDV), 0, abort_flag, p.err, p.timeout_ns);
    if (ok) {
      tc_fence_after();
      uint16_t* dst = p.dk + (static_cast<size_t>(sp.row_base) + kv_row) * row_stride + static_cast<size_t>(sp.h) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32];
        tmem_ld32(lane_addr + C::DK_COL + ch * 32, a);
        tmem_wait_ld();
        reg_fence(a);
        if (!row_dead) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(a[8 * v4 + 0]) * p.scale, __uint_as_float(a[8 * v4 + 1]) * p.scale);
            w.y = pack_bf16x2(__uint_as_float(a[8 * v4 + 2]) * p.scale, __uint_as_float(a[8 * v4 + 3]) * p.scale);
            w.z = pack_bf16x2(__uint_as_float(a[8 * v4 + 4]) * p.scale, __uint_as_float(a[8 * v4 + 5]) * p.scale);
            w.w = pack_bf16x2(__uint_as_float(a[8 * v4 + 6]) * p.scale, __uint_as_float(a[8 * v4 + 7]) * p.scale);
            reinterpret_cast<uint4*>(dst + ch * 32)[v4] = w;
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- dQ drain, dV
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    for (int ii = 0; ii < nq; ++ii) {
      const int q = (i_first + ii) * kTile + r;
      if (!wait_bounded(bar(C::B_DQFULL), ii & 1, abort_flag, p.err, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t a[D / 32][32];
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(lane_addr + C::S_COL + ch * 32, a[ch]);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) reg_fence(a[ch]);
      tc_fence_before();
      mbar_arrive(bar(C::B_DQDRAINED));
      if (q < sp.seqlen) {
        float4* dst = reinterpret_cast<float4*>(p.dq_accum + (static_cast<size_t>(sp.row_base) + q) * row_stride +
                                                static_cast<size_t>(sp.h) * D);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch)
#pragma unroll
          for (int v = 0; v < 8; ++v)
            atomicAdd(dst + ch * 8 + v,
                      make_float4(__uint_as_float(a[ch][4 * v]), __uint_as_float(a[ch][4 * v + 1]),
                                  __uint_as_float(a[ch][4 * v + 2]), __uint_as_float(a[ch][4 * v + 3])));
      }
    }
    if (ok) ok = wait_bounded(bar(C::B_DKDV), 0, abort_flag, p.err, p.timeout_ns);
    if (ok) {
      tc_fence_after();
      const int kv_row = kv0 + r;
      uint16_t* dst = p.dv + (static_cast<size_t>(sp.row_base) + kv_row) * row_stride + static_cast<size_t>(sp.h) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32];
        tmem_ld32(lane_addr + C::DV_COL + ch * 32, a);
        tmem_wait_ld();
        reg_fence(a);
        if (kv_row < sp.seqlen) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(a[8 * v4 + 0]), __uint_as_float(a[8 * v4 + 1]));
            w.y = pack_bf16x2(__uint_as_float(a[8 * v4 + 2]), __uint_as_float(a[8 * v4 + 3]));
            w.z = pack_bf16x2(__uint_as_float(a[8 * v4 + 4]), __uint_as_float(a[8 * v4 + 5]));
            w.w = pack_bf16x2(__uint_as_float(a[8 * v4 + 6]), __uint_as_float(a[8 * v4 + 7]));
            reinterpret_cast<uint4*>(dst + ch * 32)[v4] = w;
          }
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

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                         const BwdParams& p, int max_seqlen, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1) {
  using C = BwdCfg<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(fa_bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long pairs = static_cast<long long>(p.rows) * p.sv.H;
  fa_bwd_pre_kernel<D><<<static_cast<unsigned>((pairs * 32 + 255) / 256), 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 grid(p.nseq * p.sv.H, (max_seqlen + kTile - 1) / kTile);
  if (ev0 && (e = cudaEventRecord(ev0, s)) != cudaSuccess) return e;
  fa_bwd_main_kernel<D><<<grid, C::NUM_THREADS, C::SMEM_BYTES, s>>>(tq, tk, tv, tdo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev1 && (e = cudaEventRecord(ev1, s)) != cudaSuccess) return e;
  const size_t n8 = static_cast<size_t>(pairs) * D / 8;
  fa_bwd_post_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(p, n8);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int max_seqlen, cudaStream_t s,
                       cudaEvent_t main_start, cudaEvent_t main_end) {
  if (d == 64) return launch_bwd_d<64>(tq, tk, tv, tdo, p, max_seqlen, s, main_start, main_end);
  return launch_bwd_d<128>(tq, tk, tv, tdo, p, max_seqlen, s, main_start, main_end);
}

}  // namespace fa
