// Forward attention kernel for sm_103a.
//
// One CTA owns two 128-row query tiles of one (sequence, head) and streams the
// 128-key K/V tiles of that head through shared memory (query tile outer,
// key/value tile inner, O written once: "08 · FlashAttention", section 二).
// Warp roles:
//   warps 0-3, 4-7  softmax warpgroups, one per query tile; thread r of a
//                   warpgroup owns query row r (TMEM lane r), so row max and
//                   row sum need no shuffles.
//   warp 8          TMA producer (Q once, K/V through multi-stage rings).
//   warp 9          tcgen05.mma issuer.
// Per key tile j and query tile t:
//   S_t = Q_t K_jᵀ                    SMEM x SMEM -> TMEM (fp32, 128 cols)
//   softmax t: m, P = 2^(c·S − c·m_ref), l += Σ P, P as bf16 over S in TMEM
//   O_t += P_t V_j                    TMEM(A) x SMEM -> TMEM (fp32, d cols)
// The MMA order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) lets softmax of one
// query tile run while the tensor core works on the other ("LLM Systems 22",
// sections 4.1.2 and 4.2.1: overlap of GEMM and exponentials across tiles).
//
// Online softmax ("LLM Systems 22", section 3.1; "08 · FlashAttention",
// section 二) with the scale folded into the base-2 exponent
// (c = scale·log2 e) and the output kept unnormalised until the end.  The
// reference max m_ref is the first key tile's row max and is only moved when
// a later tile's row sum reaches 2^40 (P may exceed 1, by less than 2^40);
// otherwise neither a max pass nor a rescale of O in TMEM runs ("LLM Systems
// 22", section 4.2.1: an online softmax variant that skips most rescaling).
// The result is exact after the final division by l.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_kernels.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

// NQT_ query tiles per CTA: two at d = 128 (one CTA per SM, the two tiles'
// MMAs and softmaxes interleaved); one at d = 64, where a CTA's tensor memory
// (256 columns) and shared memory (~97 KB) let two CTAs share an SM, so one
// CTA's MMAs fill the tensor pipe while the other's softmax runs, and one
// CTA's prologue and epilogue overlap the other's work.
template <int D, int NQT_>
struct FwdCfg {
  static constexpr int NQT = NQT_;                      // query tiles per CTA
  static constexpr int MIN_BLOCKS = NQT == 1 ? 2 : 1;   // CTAs per SM
  static constexpr int KB = D / 64;                     // 128-byte swizzle blocks per row
  static constexpr int BLK_BYTES = kTile * 128;         // one 128-row x 64-col block
  static constexpr int TILE_BYTES = KB * BLK_BYTES;     // one 128 x D tile
  static constexpr int NSK = (D == 128 || NQT == 1) ? 3 : 4;  // K ring depth
  static constexpr int NSV = (D == 128 || NQT == 1) ? 2 : 4;  // V ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQT * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NSV * TILE_BYTES;
  // barriers: q[NQT], kfull[NSK], kempty[NSK], vfull[NSV], vempty[NSV], sfull[NQT], pfull[NQT],
  // odone[NQT], drain
  static constexpr int B_Q = 0;                         // [NQT]: query tile t landed
  static constexpr int B_KFULL = NQT;
  static constexpr int B_KEMPTY = B_KFULL + NSK;
  static constexpr int B_VFULL = B_KEMPTY + NSK;
  static constexpr int B_VEMPTY = B_VFULL + NSV;
  static constexpr int B_SFULL = B_VEMPTY + NSV;
  static constexpr int B_PFULL = B_SFULL + NQT;
  static constexpr int B_ODONE = B_PFULL + NQT;
  static constexpr int B_DRAIN = B_ODONE + NQT;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem slot, abort flag
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack to align the base to 1024
  static constexpr int NUM_WARPS = 4 * NQT + 2;
  static constexpr int NUM_THREADS = NUM_WARPS * 32;
  static constexpr int PRODUCER_WARP = 4 * NQT;
  static constexpr int MMA_WARP = 4 * NQT + 1;
  static constexpr uint32_t TMEM_COLS = NQT == 2 ? 512 : 256;
  // TMEM columns: S_t (P_t aliases its first 64 columns) and O_t.
  __host__ __device__ static constexpr uint32_t S_COL(int t) { return t * 128; }
  __host__ __device__ static constexpr uint32_t O_COL(int t) { return NQT * 128 + t * D; }
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(NQT * (128 + D) <= static_cast<int>(TMEM_COLS), "tensor memory budget");
  // CTAs sharing an SM: 228 KB of shared memory, 1 KB of it reserved per CTA.
  static_assert(MIN_BLOCKS * (SMEM_BYTES + 1024) <= 233472, "shared memory for the CTAs of one SM");
};

template <int D, int NQT_>
__global__ void __launch_bounds__(FwdCfg<D, NQT_>::NUM_THREADS, FwdCfg<D, NQT_>::MIN_BLOCKS)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
  using C = FwdCfg<D, NQT_>;
  constexpr int NQT = C::NQT;
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
  int pair, tile;
  cta_item(p.sv, pair, tile);
  if (pair >= p.sv.npairs) return;
  const SeqPos sp = seq_pos(p.sv, pair);
  // Causal: the last query tiles see the most keys, so they go first.
  const int ctile = p.causal ? p.sv.ntiles - 1 - tile : tile;
  const int q0 = ctile * kTile * NQT;
  if (q0 >= sp.seqlen) return;  // whole CTA past the end of a short packed sequence

  const int nkv_total = (sp.seqlen + kTile - 1) / kTile;
  int nkv[NQT];
  int nkv_max = 0;
#pragma unroll
  for (int t = 0; t < NQT; ++t) {
    const int qt = q0 + t * kTile;
    nkv[t] = qt >= sp.seqlen ? 0 : (p.causal ? min(nkv_total, qt / kTile + 1) : nkv_total);
    nkv_max = max(nkv_max, nkv[t]);
  }

  // TMA issue of Q and of K/V tile j into its ring slot (producer thread).
  auto load_q = [&](int t) {
    mbar_arrive_expect_tx(bar(C::B_Q + t), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_Q + t * C::TILE_BYTES + kb * C::BLK_BYTES, &tmQ, bar(C::B_Q + t), kb * 64, sp.h,
                  sp.tma_row0 + q0 + t * kTile, sp.tma_b);
  };
  auto load_k = [&](int j) {
    const int ks = j % C::NSK;
    mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_K + ks * C::TILE_BYTES + kb * C::BLK_BYTES, &tmK, bar(C::B_KFULL + ks), kb * 64,
                  sp.h, sp.tma_row0 + j * kTile, sp.tma_b);
  };
  auto load_v = [&](int j) {
    const int vs = j % C::NSV;
    mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_V + vs * C::TILE_BYTES + kb * C::BLK_BYTES, &tmV, bar(C::B_VFULL + vs), kb * 64,
                  sp.h, sp.tma_row0 + j * kTile, sp.tma_b);
  };
  // K/V tiles whose ring slots start empty: loaded by the producer as soon as
  // it has initialised the barriers, so the first loads overlap the TMEM
  // allocation and the CTA-wide barrier.
  const int preloaded = min(nkv_max, C::NSV);

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int t = 0; t < NQT; ++t) mbar_init(bar(C::B_Q + t), 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_PFULL + t), 128);
      mbar_init(bar(C::B_ODONE + t), 1);
    }
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    // In the order the first MMAs need them: Q_0 and K_0 (for S_0), then the
    // other query tiles, then V_0, so S_0 of the first key tile can start
    // before the whole set has landed.
    load_q(0);
    if (preloaded > 0) load_k(0);
#pragma unroll
    for (int t = 1; t < NQT; ++t)
      if (nkv[t] > 0) load_q(t);
    if (preloaded > 0) load_v(0);
    for (int j = 1; j < preloaded; ++j) {
      load_k(j);
      load_v(j);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::PRODUCER_WARP) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      int k_fills = preloaded, v_fills = preloaded;
      for (int j = preloaded; j < nkv_max; ++j) {
        const int ks = j % C::NSK;
        if (j >= C::NSK && !wait_bounded(bar(C::B_KEMPTY + ks), ((j / C::NSK) - 1) & 1, abort_flag, p.err,
                                         p.timeout_ns))
          break;
        load_k(j);
        ++k_fills;
        const int vs = j % C::NSV;
        if (j >= C::NSV && !wait_bounded(bar(C::B_VEMPTY + vs), ((j / C::NSV) - 1) & 1, abort_flag, p.err,
                                         p.timeout_ns))
          break;
        load_v(j);
        ++v_fills;
      }
      // Every copy this thread issued lands before the CTA may exit, whoever
      // aborted and whenever: a consumer can abort after this loop has issued
      // its last load, and a CTA that exits with a copy still writing into its
      // shared memory corrupts whatever the SM runs next.  On a clean run all
      // of these phases have completed already (the MMA thread waited on
      // them), so the waits return at once.
#pragma unroll
      for (int t = 0; t < NQT; ++t)
        if (nkv[t] > 0) wait_drain(bar(C::B_Q + t), 0, p.err, p.timeout_ns);
      for (int s = 0; s < C::NSK && s < k_fills; ++s)
        wait_drain(bar(C::B_KFULL + s), ((s + ((k_fills - 1 - s) / C::NSK) * C::NSK) / C::NSK) & 1, p.err,
                   p.timeout_ns);
      for (int s = 0; s < C::NSV && s < v_fills; ++s)
        wait_drain(bar(C::B_VFULL + s), ((s + ((v_fills - 1 - s) / C::NSV) * C::NSV) / C::NSV) & 1, p.err,
                   p.timeout_ns);
    }
  } else if (warp == C::MMA_WARP) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
      // Descriptors of the tile bases; each K16 step adds a byte offset.
      const uint64_t dQ0 = sdesc_sw128(sb + C::OFF_Q, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sb + C::OFF_V, C::BLK_BYTES, 1024);
      auto issue_s = [&](int t, int ks) {
        const uint64_t dQ = sdesc_add(dQ0, t * C::TILE_BYTES), dK = sdesc_add(dK0, ks * C::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk / 4) * C::BLK_BYTES + (kk % 4) * 32;
          mma_ss(tmem + C::S_COL(t), sdesc_add(dQ, koff), sdesc_add(dK, koff), idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int vs, bool acc) {
        const uint64_t dV = sdesc_add(dV0, vs * C::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + kk * 8, sdesc_add(dV, kk * 2048), idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_bounded(bar(C::B_KFULL + 0), 0, abort_flag, p.err, p.timeout_ns);
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        if (ok && nkv[t] > 0) {
          ok = wait_bounded(bar(C::B_Q + t), 0, abort_flag, p.err, p.timeout_ns);
          if (ok) {
            tc_fence_after();
            issue_s(t, 0);
            tc_commit(bar(C::B_SFULL + t));
          }
        }
      }
      if (ok) tc_commit(bar(C::B_KEMPTY + 0));
      for (int j = 0; ok && j < nkv_max; ++j) {
        const int vs = j % C::NSV;
        const bool next = j + 1 < nkv_max;
        const int ks1 = (j + 1) % C::NSK;
        ok = wait_bounded(bar(C::B_VFULL + vs), (j / C::NSV) & 1, abort_flag, p.err, p.timeout_ns);
        if (ok && next) ok = wait_bounded(bar(C::B_KFULL + ks1), ((j + 1) / C::NSK) & 1, abort_flag, p.err,
                                          p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (j < nkv[t]) {
            if (!wait_bounded(bar(C::B_PFULL + t), j & 1, abort_flag, p.err, p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, vs, j > 0);
            // O_t is final after its last PV: under a causal mask query tile
            // 0 sees one key tile fewer than tile 1, so its epilogue (and the
            // egress of its TMA store) overlaps tile 1's last iteration.
            if (j + 1 == nkv[t]) tc_commit(bar(C::B_ODONE + t));
          }
          if (j + 1 < nkv[t]) {
            issue_s(t, ks1);
            tc_commit(bar(C::B_SFULL + t));
          }
        }
        if (!ok) break;
        tc_commit(bar(C::B_VEMPTY + vs));
        if (next) tc_commit(bar(C::B_KEMPTY + ks1));
      }
      // Every MMA issued so far must finish before TMEM is released.
      tc_commit(bar(C::B_DRAIN));
      wait_drain(bar(C::B_DRAIN), 0, p.err, p.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int t = warp / 4;
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const int qt = q0 + t * kTile;
    const int q_row = qt + r;  // row within the sequence
    // This warp's tile's key count, computed rather than read from nkv[] with
    // a run-time index (which would put the array in local memory).
    const int nkv_t = qt >= sp.seqlen ? 0 : (p.causal ? min(nkv_total, qt / kTile + 1) : nkv_total);
    if (nkv_t > 0) {
      const float c = p.scale_log2;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
      const uint32_t tS = lane_addr + C::S_COL(t);
      const uint32_t tO = lane_addr + C::O_COL(t);
      float m_ref = -CUDART_INF_F;
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv_t; ++j) {
        if (!wait_bounded(bar(C::B_SFULL + t), j & 1, abort_flag, p.err, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(tS + ch * 32, s[ch]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) reg_fence(s[ch]);

        const int kv0 = j * kTile;
        const bool need_mask = (kv0 + kTile > sp.seqlen) || (p.causal && kv0 + kTile - 1 > qt);
        if (need_mask) {
          const int lim = p.causal ? min(sp.seqlen - 1, q_row) : sp.seqlen - 1;  // last visible key
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (kv0 + ch * 32 + i > lim) s[ch][i] = __float_as_uint(-CUDART_INF_F);
        }
        // Row max: three-input max into 4 independent partial maxima (a single
        // running max is a long dependency chain).
        auto row_max = [&]() -> float {
          float mx[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = -CUDART_INF_F;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              mx[i & 3] = fmax3(mx[i & 3], __uint_as_float(s[ch][2 * i]), __uint_as_float(s[ch][2 * i + 1]));
          return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        };
        // P = 2^(c·s − c·m_ref) as bf16 over S; returns the tile's row sum.
        // Column pairs go through the paired fp32 instructions: c·s − c·m for
        // two columns per FMA, and 4 paired partial row sums (the same 8
        // partial sums, in the same order, as one sum per column mod 8).
        auto p_pass = [&]() -> float {
          const float mc = (m_ref == -CUDART_INF_F) ? 0.f : m_ref * c;
          const uint64_t c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
          uint64_t ls2[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) ls2[k] = f2_pack(0.f, 0.f);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              f2_unpack(ffma2(f2_pack(__uint_as_float(s[ch][2 * e]), __uint_as_float(s[ch][2 * e + 1])), c2, nmc2),
                        x0, x1);
              const float p0 = ex2_approx(x0);
              const float p1 = ex2_approx(x1);
              ls2[e & 3] = fadd2(ls2[e & 3], f2_pack(p0, p1));
              pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS + ch * 16, pk);
          }
          float ls[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) f2_unpack(ls2[k], ls[2 * k], ls[2 * k + 1]);
          return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        };
        // The reference m_ref is the first key tile's row max.  Later tiles are
        // exponentiated against it without a max pass: the reference only has
        // to be common to the row, and the result is exact after the final
        // division by l ("LLM Systems 22", section 4.2.1: rescaling only when
        // needed).  A tile whose row sum leaves [0, 2^40) (a score far above
        // the reference, or a non-finite sum) takes its exact max, moves the
        // reference up, rescales O and l, and is exponentiated again: P stays
        // below 2^40 and O in fp32 range.
        if (j == 0) m_ref = row_max();
        float lt = p_pass();
        if (__any_sync(0xffffffffu, !(lt < 0x1p40f))) {
          const float m_new = fmaxf(m_ref, row_max());
          const float alpha = (m_ref == -CUDART_INF_F) ? 0.f : ex2_approx((m_ref - m_new) * c);
          m_ref = m_new;
          l *= alpha;
          // 16 columns at a time: the 128 S values of the row stay live here.
#pragma unroll 1
          for (int ch = 0; ch < D / 16; ++ch) {
            uint32_t o[16];
            tmem_ld16(tO + ch * 16, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + ch * 16, o);
          }
          tmem_wait_st();
          lt = p_pass();
        }
        l += lt;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::B_PFULL + t));
      }
      if (ok) ok = wait_bounded(bar(C::B_ODONE + t), 0, abort_flag, p.err, p.timeout_ns);
      if (ok) {
        // O_t / l, as bf16.  A warp's 32 rows (every dense tile: the map
        // clips rows past N; in a packed batch, 32 rows that do not run past
        // their sequence) are staged in the 128-byte swizzled layout over Q_t,
        // which no MMA reads any more, and written by one TMA store per 64
        // columns; a packed warp slab that ends inside its sequence is written
        // row by row (a box would overwrite the next sequence's rows).
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.0f / l : 0.f;
        const bool store = q_row < sp.seqlen;
        const bool via_tma = !p.sv.cu_seqlens || qt + 32 * wq + 32 <= sp.seqlen;
        const uint32_t stage = sb + C::OFF_Q + t * C::TILE_BYTES;
        uint16_t* orow = p.o + (static_cast<size_t>(sp.row_base + q_row) * p.sv.H + sp.h) * D;
#pragma unroll 1
        for (int cb = 0; cb < D / 64; ++cb) {  // 64 columns (one 128-byte swizzle block) per TMEM round trip
          uint32_t o[2][32];
          tmem_ld32(tO + cb * 64, o[0]);
          tmem_ld32(tO + cb * 64 + 32, o[1]);
          tmem_wait_ld();
          reg_fence(o[0]);
          reg_fence(o[1]);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {  // 16 columns (two 16-byte chunks) at a time
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[ch / 2][(ch % 2) * 16 + 2 * e]) * inv_l,
                                 __uint_as_float(o[ch / 2][(ch % 2) * 16 + 2 * e + 1]) * inv_l);
            if (via_tma) {
              const uint32_t rowaddr = stage + cb * C::BLK_BYTES + r * 128;
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const uint32_t chunk = (ch * 2 + u) ^ (r & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowaddr + chunk * 16), "r"(w[4 * u]),
                             "r"(w[4 * u + 1]), "r"(w[4 * u + 2]), "r"(w[4 * u + 3])
                             : "memory");
              }
            } else if (store) {
              uint4* dst = reinterpret_cast<uint4*>(orow + cb * 64 + ch * 16);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
        if (store) {
          const float lse = l > 0.f ? (m_ref * c + log2f(l)) * kLn2 : -CUDART_INF_F;
          p.lse[(static_cast<size_t>(sp.bs) * p.sv.H + sp.h) * p.sv.lse_stride + q_row] = lse;
        }
        if (via_tma) {
          // Each warp stores its own 32 rows (a 32-row box whose 1024-byte
          // swizzle atoms line up with the staged rows), so no thread waits
          // for the rest of the tile to be staged.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && qt + 32 * wq < sp.seqlen) {
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_store_4d(&tmO, stage + kb * C::BLK_BYTES + wq * 4096, kb * 64, sp.h, sp.tma_row0 + qt + 32 * wq,
                           sp.tma_b);
            bulk_commit_group();
            // The stage may be released once the copies have read it; their
            // global writes complete before the grid does.
            bulk_wait_group_read0();
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

template <int D, int NQT>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                         const FwdParams& p, int nseq, int max_seqlen, cudaStream_t s) {
  using C = FwdCfg<D, NQT>;
  static SmemLimit smem_limit;
  cudaError_t e = smem_limit.ensure(reinterpret_cast<const void*>(fa_fwd_kernel<D, NQT>), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = current_sm_count(sms);
  if (e != cudaSuccess) return e;
  FwdParams pl = p;
  pl.sv.npairs = nseq * p.sv.H;
  pl.sv.ntiles = (max_seqlen + kTile * C::NQT - 1) / (kTile * C::NQT);
  pl.sv.pair_group = pair_group_size(pl.sv.npairs, pl.sv.ntiles, sms * C::MIN_BLOCKS);
  const long long ctas = grid_ctas(pl.sv.npairs, pl.sv.ntiles, pl.sv.pair_group);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_kernel<D, NQT><<<static_cast<unsigned>(ctas), C::NUM_THREADS, C::SMEM_BYTES, s>>>(tq, tk, tv, to, pl);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, int nseq, int max_seqlen, cudaStream_t s) {
  if (d == 64) return launch_fwd_d<64, 1>(tq, tk, tv, to, p, nseq, max_seqlen, s);
  return launch_fwd_d<128, 2>(tq, tk, tv, to, p, nseq, max_seqlen, s);
}

}  // namespace fa
