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
//                dQ_i is drained from TMEM through shared memory and added to
//                the fp32 accumulator by TMA bulk reduce-adds (other key tiles
//                add to the same rows).
//   fa_bwd_post  dQ = bf16(scale · dQ_accum).
// Each launch may start while the previous one finishes (programmatic
// dependent launch) and waits for it before touching what it wrote.
// Warp roles in fa_bwd_main: warps 0-7 (two warpgroups, each owning half of
// the query columns of a tile; thread r owns key row r = TMEM lane r)
// recompute P and dS, drain dQ and write dK / dV; warp 8 issues TMA; warp 9
// issues tcgen05.mma.
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
// fa_bwd_pre: D/8 threads per (row, head), 16 bytes of O and of dO each (two
// 16-byte loads in flight per thread, enough to keep HBM busy at one load
// round trip per thread).
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
  grid_launch_dependents();  // the main kernel's prologue and first MMAs need nothing from here
  constexpr int TPR = D / 8;  // threads per (row, head); rows do not straddle warps (TPR divides 32)
  static_assert(32 % TPR == 0, "a (row, head) lies within one warp");
  const int H = p.sv.H;
  const long long total = static_cast<long long>(p.rows) * H;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rh = tid / TPR;  // (row, head) = row·H + head
  const int part = static_cast<int>(tid % TPR);
  const bool live = rh < total;
  float acc = 0.f;
  if (live) {
    const size_t base = static_cast<size_t>(rh) * D + part * 8;  // [rows, H, d] element offset
    const uint4 o = *reinterpret_cast<const uint4*>(p.o + base);
    const uint4 d = *reinterpret_cast<const uint4*>(p.dout + base);
    acc = bf16lo_to_f32(o.x) * bf16lo_to_f32(d.x) + bf16hi_to_f32(o.x) * bf16hi_to_f32(d.x) +
          bf16lo_to_f32(o.y) * bf16lo_to_f32(d.y) + bf16hi_to_f32(o.y) * bf16hi_to_f32(d.y) +
          bf16lo_to_f32(o.z) * bf16lo_to_f32(d.z) + bf16hi_to_f32(o.z) * bf16hi_to_f32(d.z) +
          bf16lo_to_f32(o.w) * bf16lo_to_f32(d.w) + bf16hi_to_f32(o.w) * bf16hi_to_f32(d.w);
    float4* z = reinterpret_cast<float4*>(p.dq_accum + base);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // Every lane takes part in the shuffles (lanes past the end add zeros).
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && part == 0) {
    const int g = static_cast<int>(rh / H), h = static_cast<int>(rh - (rh / H) * H);
    int bs, local;
    locate_row(p.sv, p.nseq, g, bs, local);
    p.dpsum[(static_cast<size_t>(bs) * H + h) * p.sv.lse_stride + local] = acc;
  }
}

// ----------------------------------------------------------------------------
// fa_bwd_post: dQ = bf16(scale · accumulator), 8 elements per thread.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const BwdParams p, size_t n8) {
  grid_dependency_wait();    // every reduce-add of the main kernel has landed
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
// TMEM holds dV and dK (d columns each) for the whole loop plus two 128-column
// regions with fixed roles:
//   X: Sᵀ_i, then Pᵀ_i as bf16 (the A operand of dV_i)
//   Y: dPᵀ_i, then dQ_i
// dSᵀ_i goes to shared memory only: it is the A operand of both dQ_i (read
// MN-major, as dS) and dK_i (read K-major, as dSᵀ).  MMA order per tile:
// dV_i, Sᵀ_{i+1}, dQ_i, dK_i, dPᵀ_{i+1}.  Sᵀ_{i+1} overwrites Pᵀ_i right
// after dV_i has read it, so the compute warps form Pᵀ_{i+1} while the tensor
// pipe runs dQ_i and dK_i; dQ_i comes before dK_i so that its drain starts as
// early as possible; dPᵀ_{i+1} overwrites dQ_i once the drain warps have read
// it out of TMEM.  (MMAs issued by one thread execute in issue order, so each
// overwrite follows the read before it.)
//
// Shared memory and the dQ read-out.  A tile's fp32 dQ (64 KB at d = 128)
// leaves the SM through bulk reduce-adds at the SM's reduction egress rate
// (about 25 bytes per clock, measured alike for one SM and for all of them,
// and shared by the TMA and vector-atomic paths), so its read-out lasts about
// as long as the tile's five GEMMs, and whatever shared memory holds it is
// tied up meanwhile.  dQ is therefore staged in a buffer of its own (STG),
// never over a Q/dO ring slot that the next tiles' loads need:
//   d = 128: the dS operand of the dQ GEMM is written over the tile's dO
//            (consumed once dPᵀ_i and dV_i have completed), which frees the
//            32 KB that a separate dS buffer would take for STG; dQ columns
//            0-63 go to STG and columns 64-127 over that dS.  A slot's Q is
//            reloaded as soon as dK_i has read it, its dO once the half of dQ
//            over it has been read out.
//   d = 64:  a separate dS buffer and a 32 KB STG that holds all of dQ.
template <int D>
struct BwdCfg {
  static constexpr bool DS_IN_DO = (D == 128);         // dS written over the tile's consumed dO
  static constexpr int KB = D / 64;
  static constexpr int BLK_BYTES = kTile * 128;        // 128 rows x 64 bf16
  static constexpr int TILE_BYTES = KB * BLK_BYTES;    // 128 x D bf16
  static constexpr int NSQ = (D == 128) ? 2 : 3;       // Q / dO ring depth
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + NSQ * TILE_BYTES;
  // dSᵀ, 128 key rows x 128 queries in two 64-query blocks (d = 64 only)
  static constexpr int OFF_DS = OFF_DO + NSQ * TILE_BYTES;
  static constexpr int OFF_STG = OFF_DS + (DS_IN_DO ? 0 : 2 * BLK_BYTES);  // dQ staging, 32 KB
  static constexpr int STG_BYTES = 32768;
  static constexpr int OFF_STAT = OFF_STG + STG_BYTES;  // [2][2][128] fp32: log2e·LSE and D
  static constexpr int OFF_BAR = OFF_STAT + 2 * 2 * kTile * 4;
  static constexpr int B_K = 0;
  static constexpr int B_V = 1;
  static constexpr int B_QFULL = 2;
  static constexpr int B_DOFULL = B_QFULL + NSQ;
  // [NSQ]: dK of the slot's tile has read its Q and dS (both the slot's Q and,
  // at d = 128, the dS over its dO may be overwritten)
  static constexpr int B_QFREE = B_DOFULL + NSQ;
  static constexpr int B_DOFREE = B_QFREE + NSQ;       // [NSQ] (d = 64): dV of the slot's tile has read its dO
  static constexpr int B_STAGED = B_DOFREE + NSQ;      // the drain warps have staged a tile's dQ
  static constexpr int B_STGFREE = B_STAGED + 1;       // the reduces have read STG
  static constexpr int B_DVDONE = B_STGFREE + 1;       // (d = 128) dV_i has read dO_i: dS may go over it
  static constexpr int B_SFULL = B_DVDONE + 1;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_PREADY = B_DPFULL + 1;
  static constexpr int B_DSREADY = B_PREADY + 1;
  static constexpr int B_DQFULL = B_DSREADY + 1;
  static constexpr int B_DQDRAINED = B_DQFULL + 1;
  static constexpr int B_DKDV = B_DQDRAINED + 1;
  static constexpr int B_DRAIN = B_DKDV + 1;
  static constexpr int B_STAT = B_DRAIN + 1;           // [2]: row statistics of a query tile staged
  static constexpr int NBAR = B_STAT + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // Whatever is left of the 227 KB opt-in limit is alignment slack.
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024 <= 232448) ? SMEM_USED + 1024 : 232448;
  static constexpr int NCHT = D / 32;                  // 32-column dQ chunks per row
  static constexpr int NCH_STG = 2;                    // chunks 0, 1 are staged in STG
  static_assert(kTile * NCH_STG * 32 * 4 == STG_BYTES, "STG holds two 32-column chunks of a tile");
  // Byte offset of the staging slice (32 rows x 32 fp32 columns, 4 KB,
  // 128-byte swizzled) of dQ rows 32·wq .. +31, columns 32·c .. +31, for the
  // tile in ring slot qs.
  __host__ __device__ static constexpr uint32_t dq_slice(int qs, int c, int wq) {
    return c < NCH_STG ? OFF_STG + (c * 4 + wq) * 4096
                       : OFF_DO + qs * TILE_BYTES + ((c - NCH_STG) * 4 + wq) * 4096;
  }
  // Base of the dSᵀ tile of the query tile in ring slot qs.
  __host__ __device__ static constexpr uint32_t ds_base(int qs) {
    return DS_IN_DO ? OFF_DO + qs * TILE_BYTES : OFF_DS;
  }
  static constexpr int NUM_COMPUTE = 256;              // warps 0-7: two warpgroups
  static constexpr int NUM_DRAIN = 128;                // warps 10-13: one per TMEM lane quarter
  // Warps 14-15 only complete the fourth warpgroup, so that registers can be
  // moved per warpgroup: the CTA launches with LAUNCH_REGS registers a thread
  // (65536 / NUM_THREADS in the allocation's steps of 8: 128); the two
  // compute warpgroups take REG_COMPUTE, the other two give back to
  // REG_OTHER.  The increases are served from the registers the CTA launched
  // with, so the split must fit in them or an increase waits forever.
  static constexpr int NUM_THREADS = 512;
  static constexpr int LAUNCH_REGS = (65536 / NUM_THREADS) & ~7;
  static constexpr int REG_COMPUTE = 160;
  static constexpr int REG_OTHER = 96;
  static_assert(NUM_COMPUTE * REG_COMPUTE + (NUM_THREADS - NUM_COMPUTE) * REG_OTHER <= NUM_THREADS * LAUNCH_REGS,
                "register split exceeds the CTA's launch allocation");
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int DRAIN_WARP0 = 10;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t DV_COL = 0;
  static constexpr uint32_t DK_COL = D;
  static constexpr uint32_t R_COL = 2 * D;             // X = R_COL, Y = R_COL + 128
  static_assert(SMEM_USED <= 232448, "shared memory budget");
  static_assert(!DS_IN_DO || TILE_BYTES == 2 * BLK_BYTES, "dSᵀ (two 64-query blocks) fits over a dO tile");
  static_assert(!DS_IN_DO || (NCHT - NCH_STG) * 4 * 4096 <= TILE_BYTES, "dQ half fits over a dO tile");
};

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::NUM_THREADS, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                       const __grid_constant__ CUtensorMap tmDV, const BwdParams p) {
  using C = BwdCfg<D>;
  grid_launch_dependents();  // the dQ conversion may be scheduled; it waits for this grid to finish
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
  float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);  // [buf][0: log2e·LSE, 1: D][128]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int pair, j;                        // j: key tile; heavy (small j) tiles first under a causal mask
  cta_item(p.sv, pair, j);
  if (pair >= p.sv.npairs) return;
  const SeqPos sp = seq_pos(p.sv, pair);
  const int kv0 = j * kTile;
  if (kv0 >= sp.seqlen) return;
  const int nq_total = (sp.seqlen + kTile - 1) / kTile;
  const int i_first = p.causal ? j : 0;
  const int nq = nq_total - i_first;

  // TMA issue of query tile ii's Q and dO into ring slot ii % NSQ (producer
  // thread).
  auto load_q = [&](int ii) {
    const int qs = ii % C::NSQ;
    const int qrow = sp.tma_row0 + (i_first + ii) * kTile;
    mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_Q + qs * C::TILE_BYTES + kb * C::BLK_BYTES, &tmQ, bar(C::B_QFULL + qs), kb * 64, sp.h,
                  qrow, sp.tma_b);
  };
  auto load_do = [&](int ii) {
    const int qs = ii % C::NSQ;
    const int qrow = sp.tma_row0 + (i_first + ii) * kTile;
    mbar_arrive_expect_tx(bar(C::B_DOFULL + qs), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_DO + qs * C::TILE_BYTES + kb * C::BLK_BYTES, &tmdO, bar(C::B_DOFULL + qs), kb * 64,
                  sp.h, qrow, sp.tma_b);
  };
  // K, V and the query tiles whose ring slots start empty are loaded by the
  // producer as soon as it has initialised the barriers, so the first loads
  // overlap the TMEM allocation and the CTA-wide barrier.
  const int preloaded = min(nq, C::NSQ);

  if (warp == C::PRODUCER_WARP && lane == 0) {
    mbar_init(bar(C::B_K), 1);
    mbar_init(bar(C::B_V), 1);
    for (int s = 0; s < C::NSQ; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1);
      mbar_init(bar(C::B_DOFULL + s), 1);
      mbar_init(bar(C::B_QFREE + s), 1);
      mbar_init(bar(C::B_DOFREE + s), 1);
    }
    mbar_init(bar(C::B_STAGED), C::NUM_DRAIN);
    mbar_init(bar(C::B_STGFREE), 1);
    mbar_init(bar(C::B_DVDONE), 1);
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PREADY), C::NUM_COMPUTE);
    mbar_init(bar(C::B_DSREADY), C::NUM_COMPUTE);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQDRAINED), C::NUM_DRAIN);
    mbar_init(bar(C::B_DKDV), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    mbar_init(bar(C::B_STAT + 0), C::NUM_COMPUTE);
    mbar_init(bar(C::B_STAT + 1), C::NUM_COMPUTE);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmDK);
    tma_prefetch_desc(&tmDV);
    // In the order the first MMAs need them: K and Q_0 (Sᵀ_0), then V and
    // dO_0 (dPᵀ_0), then the rest of the ring.
    mbar_arrive_expect_tx(bar(C::B_K), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_K + kb * C::BLK_BYTES, &tmK, bar(C::B_K), kb * 64, sp.h, sp.tma_row0 + kv0, sp.tma_b);
    if (preloaded > 0) load_q(0);
    mbar_arrive_expect_tx(bar(C::B_V), C::TILE_BYTES);
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_4d(sb + C::OFF_V + kb * C::BLK_BYTES, &tmV, bar(C::B_V), kb * 64, sp.h, sp.tma_row0 + kv0, sp.tma_b);
    if (preloaded > 0) load_do(0);
    for (int ii = 1; ii < preloaded; ++ii) {
      load_q(ii);
      load_do(ii);
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
  const size_t stat_base = (static_cast<size_t>(sp.bs) * p.sv.H + sp.h) * p.sv.lse_stride;
  const size_t row_stride = static_cast<size_t>(p.sv.H) * D;  // elements between consecutive rows

  if (warp == C::PRODUCER_WARP) {
    // ---------------------------------------------------------------- TMA
    setmaxnreg_dec<C::REG_OTHER>();
    if (lane == 0) {
      // Per query tile t (ring slot s): reload Q of tile t + NSQ into s once
      // dK_t has read Q_t; add the staged dQ_t into the accumulator (TMA bulk
      // reduce-adds, the STG part first, so that the drain of tile t + 1 can
      // reuse STG); reload dO of tile t + NSQ once nothing reads the slot's
      // dO region any more (d = 128: the half of dQ_t staged over it has been
      // read; d = 64: dV_t has read dO_t).
      auto reduce_chunks = [&](int t, int c_lo, int c_hi) {
        const int qs = t % C::NSQ;
        const int q0 = (i_first + t) * kTile;
#pragma unroll 1
        for (int wq = 0; wq < 4; ++wq) {
#pragma unroll
          for (int c = c_lo; c < c_hi; ++c)
            tma_reduce_add_3d(&tmDQ, sb + C::dq_slice(qs, c, wq), 32 * c, sp.h, sp.row_base + q0 + 32 * wq);
        }
        bulk_commit_group();
      };
      // The first reduce-add needs the accumulator zeroed by the pre-pass
      // (plain stores, possibly still running when this kernel started).
      grid_dependency_wait();
      fence_proxy_async_global();
      int q_fills = preloaded, do_fills = preloaded;
      for (int t = 0; t < nq; ++t) {
        const int s = t % C::NSQ;
        const int nxt = t + C::NSQ;
        const uint32_t ph = (t / C::NSQ) & 1;
        if (nxt < nq) {
          if (!wait_bounded(bar(C::B_QFREE + s), ph, abort_flag, p.err, p.timeout_ns)) break;
          load_q(nxt);
          ++q_fills;
        }
        if (!wait_bounded(bar(C::B_STAGED), t & 1, abort_flag, p.err, p.timeout_ns)) break;
        reduce_chunks(t, 0, C::NCH_STG);
        if constexpr (C::NCHT > C::NCH_STG) {
          reduce_chunks(t, C::NCH_STG, C::NCHT);
          bulk_wait_group_read<1>();   // STG has been read
        } else {
          bulk_wait_group_read0();
        }
        mbar_arrive(bar(C::B_STGFREE));
        if (nxt < nq) {
          if constexpr (C::DS_IN_DO) {
            bulk_wait_group_read0();   // the half of dQ over the dO region has been read
          } else {
            if (!wait_bounded(bar(C::B_DOFREE + s), ph, abort_flag, p.err, p.timeout_ns)) break;
          }
          load_do(nxt);
          ++do_fills;
        }
      }
      bulk_wait_group_read0();   // every reduce has read its source; the adds land before the grid ends
      // Every load this thread issued lands before the CTA may exit, whoever
      // aborted and whenever (on a clean run these phases have all completed).
      wait_drain(bar(C::B_K), 0, p.err, p.timeout_ns);
      wait_drain(bar(C::B_V), 0, p.err, p.timeout_ns);
      for (int s = 0; s < C::NSQ && s < q_fills; ++s)
        wait_drain(bar(C::B_QFULL + s), ((s + ((q_fills - 1 - s) / C::NSQ) * C::NSQ) / C::NSQ) & 1, p.err,
                   p.timeout_ns);
      for (int s = 0; s < C::NSQ && s < do_fills; ++s)
        wait_drain(bar(C::B_DOFULL + s), ((s + ((do_fills - 1 - s) / C::NSQ) * C::NSQ) / C::NSQ) & 1, p.err,
                   p.timeout_ns);
    }
  } else if (warp == C::MMA_WARP) {
    // ---------------------------------------------------------------- MMA
    setmaxnreg_dec<C::REG_OTHER>();
    if (lane == 0) {
      constexpr uint32_t idesc_sp = idesc_bf16(128, 128, false, false);   // Sᵀ, dPᵀ
      constexpr uint32_t idesc_kv = idesc_bf16(128, D, false, true);      // dV (A from TMEM), dK
      constexpr uint32_t idesc_q = idesc_bf16(128, D, true, true);        // dQ (A = dS, MN-major)
      auto region = [&](int r) -> uint32_t { return tmem + C::R_COL + (r & 1) * 128; };
      // Tile-base descriptors, K-major (k steps of 32 bytes within a
      // 128-byte row) and MN-major (k steps of 16 rows = 2048 bytes).
      const uint64_t kmK = sdesc_sw128(sb + C::OFF_K, 16, 1024), kmV = sdesc_sw128(sb + C::OFF_V, 16, 1024);
      const uint64_t kmQ = sdesc_sw128(sb + C::OFF_Q, 16, 1024), kmDO = sdesc_sw128(sb + C::OFF_DO, 16, 1024);
      const uint64_t mnQ = sdesc_sw128(sb + C::OFF_Q, C::BLK_BYTES, 1024);
      const uint64_t mnDO = sdesc_sw128(sb + C::OFF_DO, C::BLK_BYTES, 1024);
      const uint64_t mnK = sdesc_sw128(sb + C::OFF_K, C::BLK_BYTES, 1024);
      auto issue_sp = [&](uint32_t dst, uint64_t a, uint64_t b) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk / 4) * C::BLK_BYTES + (kk % 4) * 32;
          mma_ss(dst, sdesc_add(a, koff), sdesc_add(b, koff), idesc_sp, kk > 0);
        }
      };
      bool ok = wait_bounded(bar(C::B_K), 0, abort_flag, p.err, p.timeout_ns) &&
                wait_bounded(bar(C::B_QFULL + 0), 0, abort_flag, p.err, p.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_sp(region(0), kmK, kmQ);                                     // Sᵀ_0 -> X
        tc_commit(bar(C::B_SFULL));
        ok = wait_bounded(bar(C::B_V), 0, abort_flag, p.err, p.timeout_ns) &&
             wait_bounded(bar(C::B_DOFULL + 0), 0, abort_flag, p.err, p.timeout_ns);
      }
      if (ok) {
        tc_fence_after();
        issue_sp(region(1), kmV, kmDO);                                    // dPᵀ_0 -> Y
        tc_commit(bar(C::B_DPFULL));
      }
      const uint32_t tX = region(0), tY = region(1);
      for (int ii = 0; ok && ii < nq; ++ii) {
        const int qs = ii % C::NSQ;
        const uint64_t bQ = sdesc_add(mnQ, qs * C::TILE_BYTES), bdO = sdesc_add(mnDO, qs * C::TILE_BYTES);
        const uint64_t aDS = sdesc_sw128(sb + C::ds_base(qs), C::BLK_BYTES, 1024);  // dS, MN-major
        const uint64_t kDS = sdesc_sw128(sb + C::ds_base(qs), 16, 1024);            // dSᵀ, K-major
        const bool next = ii + 1 < nq;
        const int qs1 = (ii + 1) % C::NSQ;
        const uint32_t ph1 = ((ii + 1) / C::NSQ) & 1;
        ok = wait_bounded(bar(C::B_PREADY), ii & 1, abort_flag, p.err, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)  // dV += Pᵀ dO_i (Pᵀ packed in X)
          mma_ts(tmem + C::DV_COL, tX + (kk / 4) * 64 + (kk % 4) * 8, sdesc_add(bdO, kk * 2048), idesc_kv,
                 (ii > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(C::DS_IN_DO ? C::B_DVDONE : C::B_DOFREE + qs));  // dO_i read: dS (or the next dO) may go there
        if (next) {
          ok = wait_bounded(bar(C::B_QFULL + qs1), ph1, abort_flag, p.err, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          issue_sp(tX, kmK, sdesc_add(kmQ, qs1 * C::TILE_BYTES));               // Sᵀ_{i+1} -> X (after dV_i)
          tc_commit(bar(C::B_SFULL));
        }
        ok = wait_bounded(bar(C::B_DSREADY), ii & 1, abort_flag, p.err, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)  // dQ_i = dS K_j -> Y (dPᵀ_i read by the compute warps)
          mma_ss(tY, sdesc_add(aDS, kk * 2048), sdesc_add(mnK, kk * 2048), idesc_q, kk > 0);
        tc_commit(bar(C::B_DQFULL));
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {  // dK += dSᵀ Q_i (dSᵀ K-major from shared memory)
          const uint32_t koff = (kk / 4) * C::BLK_BYTES + (kk % 4) * 32;
          mma_ss(tmem + C::DK_COL, sdesc_add(kDS, koff), sdesc_add(bQ, kk * 2048), idesc_kv,
                 (ii > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(C::B_QFREE + qs));          // Q_i and dS_i read: the slot may be reused
        if (next) {
          ok = wait_bounded(bar(C::B_DQDRAINED), ii & 1, abort_flag, p.err, p.timeout_ns);
          if (!ok) break;
          ok = wait_bounded(bar(C::B_DOFULL + qs1), ph1, abort_flag, p.err, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          issue_sp(tY, kmV, sdesc_add(kmDO, qs1 * C::TILE_BYTES));              // dPᵀ_{i+1} -> Y
          tc_commit(bar(C::B_DPFULL));
        }
      }
      if (ok) tc_commit(bar(C::B_DKDV));
      tc_commit(bar(C::B_DRAIN));
      wait_drain(bar(C::B_DRAIN), 0, p.err, p.timeout_ns);
    }
  } else if (warp >= C::DRAIN_WARP0 + 4) {
    setmaxnreg_dec<C::REG_OTHER>();        // warps 14-15: no role
  } else if (warp >= C::DRAIN_WARP0) {
    // ---------------------------------------------------------------- dQ drain
    setmaxnreg_dec<C::REG_OTHER>();
    // One warp per TMEM lane quarter wq (dQ rows 32·wq .. +31 of the query
    // tile; thread = row).  Once dQ_i has completed, copy the rows from TMEM
    // into the 128-byte swizzled staging slices, two 32-column chunks at a
    // time: first, once the reduces of tile i − 1 have read STG, the chunks
    // that go to STG; then (d = 128) the other chunks, which go over the
    // tile's dS: they are read out of TMEM at once, so the TMEM region is
    // released to the MMA warp, and stored once dK_i has finished reading dS.
    // Then the slices are handed to the TMA producer, which adds them into
    // the accumulator.  Rows past the sequence end carry exact zeros (their
    // P, hence dS, is 0).
    const int wq = warp & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    auto stage_chunk = [&](const uint32_t (&v)[32], uint32_t slice) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t chunk = u ^ (lane & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(slice + lane * 128 + chunk * 16), "r"(v[4 * u]),
                     "r"(v[4 * u + 1]), "r"(v[4 * u + 2]), "r"(v[4 * u + 3])
                     : "memory");
      }
    };
    auto load_pair = [&](uint32_t rs, int c0, uint32_t (&a)[2][32]) {
      tmem_ld32(rs + 32 * c0, a[0]);
      tmem_ld32(rs + 32 * (c0 + 1), a[1]);
      tmem_wait_ld();
      reg_fence(a[0]);
      reg_fence(a[1]);
    };
    static_assert(C::NCHT - C::NCH_STG <= 2, "at most one chunk pair is staged over dS");
    for (int ii = 0; ii < nq; ++ii) {
      const uint32_t rs = lane_addr + C::R_COL + 128;  // dQ_i in region Y
      if (!wait_bounded(bar(C::B_DQFULL), ii & 1, abort_flag, p.err, p.timeout_ns)) break;
      tc_fence_after();
      const int qs = ii % C::NSQ;
      if (ii > 0 && !wait_bounded(bar(C::B_STGFREE), (ii - 1) & 1, abort_flag, p.err, p.timeout_ns)) break;
      uint32_t a[2][32];
#pragma unroll
      for (int c0 = 0; c0 < C::NCH_STG; c0 += 2) {
        load_pair(rs, c0, a);
        stage_chunk(a[0], sb + C::dq_slice(qs, c0, wq));
        stage_chunk(a[1], sb + C::dq_slice(qs, c0 + 1, wq));
      }
      if constexpr (C::NCHT > C::NCH_STG) {
        if (!wait_bounded(bar(C::B_QFREE + qs), (ii / C::NSQ) & 1, abort_flag, p.err, p.timeout_ns)) break;
        load_pair(rs, C::NCH_STG, a);
        stage_chunk(a[0], sb + C::dq_slice(qs, C::NCH_STG, wq));
        stage_chunk(a[1], sb + C::dq_slice(qs, C::NCH_STG + 1, wq));
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DQDRAINED));
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_STAGED));
    }
  } else {
    // ---------------------------------------------------------------- P, dS
    setmaxnreg_inc<C::REG_COMPUTE>();
    // Warpgroup g owns query columns 64g .. 64g+63 of Sᵀ / dPᵀ; thread r of a
    // warpgroup owns TMEM lane r (key row r).  The row statistics of query
    // tile i+1 are loaded from global memory during tile i and published,
    // through a double-buffered shared array and an mbarrier, right after
    // dS_i, so the wait for them at the start of tile i+1 rarely blocks.
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;          // key row of Sᵀ / dPᵀ
    const int kv_row = kv0 + r;
    const bool row_dead = kv_row >= sp.seqlen;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float c = p.scale_log2;
    // LSE (warpgroup 0; +inf past the sequence end, so P = 0 there) or D
    // (warpgroup 1) of query row r of tile ii, as loaded: the value is first
    // used a whole tile later, when it is published, so nothing waits for the
    // load before then (scaling it by log2 e here would stall the warp for
    // the load's latency on every tile).
    auto load_stat = [&](int ii) -> float {
      const int q = (i_first + ii) * kTile + r;
      if (q >= sp.seqlen) return g == 0 ? CUDART_INF_F : 0.f;
      return __ldg((g == 0 ? p.lse : p.dpsum) + stat_base + q);
    };
    // Both warpgroups read all 128 entries of a tile (log2e·LSE and D):
    // publish them through an mbarrier (a bounded wait, unlike a named
    // barrier, so an abort cannot hang).  Buffer ii & 1 was last read during
    // tile ii - 2, which every thread has finished once it has passed tile
    // ii - 1's wait.
    auto publish_stat = [&](int ii, float v) {
      float* buf = stat + (ii & 1) * 256;
      buf[g * 128 + r] = g == 0 ? v * kLog2e : v;
      mbar_arrive(bar(C::B_STAT + (ii & 1)));
    };
    grid_dependency_wait();  // D comes from the pre-pass
    if (nq > 0) publish_stat(0, load_stat(0));
    // stat_next: tile ii + 1's value, published at the end of tile ii; the
    // load of tile ii + 2's is issued at the top of tile ii, before this
    // thread's shared-memory stores of the tile (a load queued behind them
    // waits for them to drain).
    float stat_next = nq > 1 ? load_stat(1) : 0.f;
    bool ok = true;
    for (int ii = 0; ii < nq; ++ii) {
      const float stat_after = ii + 2 < nq ? load_stat(ii + 2) : 0.f;
      const int qi = i_first + ii;
      const int q0 = qi * kTile;
      const uint32_t rs = lane_addr + C::R_COL;        // region X: Sᵀ, Pᵀ
      const uint32_t rp = lane_addr + C::R_COL + 128;  // region Y: dPᵀ
      const float* lse2 = stat + (ii & 1) * 256;
      const float* dsum = lse2 + 128;
      if (!wait_bounded(bar(C::B_STAT + (ii & 1)), (ii >> 1) & 1, abort_flag, p.err, p.timeout_ns)) {
        ok = false;
        break;
      }
      const bool need_mask = row_dead || (p.causal && qi == j);
      // ---- Pᵀ = 2^(c·Sᵀ − log2e·LSE) for this warpgroup's 64 query columns
      if (!wait_bounded(bar(C::B_SFULL), ii & 1, abort_flag, p.err, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pr[2][32];
      tmem_ld32(rs + 64 * g, pr[0]);
      tmem_ld32(rs + 64 * g + 32, pr[1]);
      tmem_wait_ld();
      reg_fence(pr[0]);
      reg_fence(pr[1]);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t pk[16];
        // Two copies of the loop: the test of the mask would otherwise cost a
        // compare and a select per element on every tile, not only on the
        // diagonal one and past the sequence end.
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = 64 * g + 32 * ch + e;
            float pe = ex2_approx(fmaf(__uint_as_float(pr[ch][e]), c, -lse2[col]));
            if (row_dead || q0 + col < kv_row) pe = 0.f;
            pr[ch][e] = __float_as_uint(pe);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = 64 * g + 32 * ch + e;
            pr[ch][e] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(pr[ch][e]), c, -lse2[col])));
          }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(pr[ch][2 * e]), __uint_as_float(pr[ch][2 * e + 1]));
        tmem_st16(rs + 64 * g + 16 * ch, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::B_PREADY));
      // ---- dSᵀ = Pᵀ ∘ (dPᵀ − D)
      if (!wait_bounded(bar(C::B_DPFULL), ii & 1, abort_flag, p.err, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dSᵀ row r, this warpgroup's 64 query columns -> the swizzled SMEM
      // block g (the A operand of dQ_i, MN-major, and of dK_i, K-major); at
      // d = 128 that block lies over the tile's dO, which dV_i must have
      // finished reading first.
      const uint32_t rowaddr = sb + C::ds_base(ii % C::NSQ) + g * C::BLK_BYTES + r * 128;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t dp[32];
        tmem_ld32(rp + 64 * g + 32 * ch, dp);
        tmem_wait_ld();
        reg_fence(dp);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = 64 * g + 32 * ch + 2 * e;
          const float d0 = __uint_as_float(pr[ch][2 * e]) * (__uint_as_float(dp[2 * e]) - dsum[col]);
          const float d1 = __uint_as_float(pr[ch][2 * e + 1]) * (__uint_as_float(dp[2 * e + 1]) - dsum[col + 1]);
          dk[e] = pack_bf16x2(d0, d1);
        }
        if constexpr (C::DS_IN_DO) {
          if (ch == 0 && !wait_bounded(bar(C::B_DVDONE), ii & 1, abort_flag, p.err, p.timeout_ns)) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t chunk = (ch * 4 + u) ^ (r & 7);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowaddr + chunk * 16), "r"(dk[4 * u]),
                       "r"(dk[4 * u + 1]), "r"(dk[4 * u + 2]), "r"(dk[4 * u + 3])
                       : "memory");
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSREADY));
      if (ii + 1 < nq) publish_stat(ii + 1, stat_next);
      stat_next = stat_after;
    }
    if (ok) ok = wait_bounded(bar(C::B_DKDV), 0, abort_flag, p.err, p.timeout_ns);
    if (ok) {
      // Warpgroup 0 writes dK (scaled), warpgroup 1 writes dV.  Every MMA
      // has completed, so the K and V tiles in shared memory are free: each
      // warp stages its 32 rows there (128-byte swizzled, as they were
      // loaded) and stores them with one TMA store per 64 columns.  (Plain
      // stores, each warp instruction touching 32 rows 4 KB apart, took
      // ≈ 4 µs per CTA for these 64 KB.)  A packed 32-row slab that runs past
      // its sequence's end is written row by row (a box would overwrite the
      // next sequence's rows).
      tc_fence_after();
      const float mul = g == 0 ? p.scale : 1.0f;
      const bool via_tma = !p.sv.cu_seqlens || kv0 + 32 * wq + 32 <= sp.seqlen;
      const uint32_t stage = sb + (g == 0 ? C::OFF_K : C::OFF_V);
      uint16_t* dst = (g == 0 ? p.dk : p.dv) + (static_cast<size_t>(sp.row_base) + kv_row) * row_stride +
                      static_cast<size_t>(sp.h) * D;
      const uint32_t src = lane_addr + (g == 0 ? C::DK_COL : C::DV_COL);
#pragma unroll 1
      for (int cb = 0; cb < D / 64; ++cb) {  // 64 columns (one 128-byte swizzle block) per TMEM round trip
        uint32_t v[2][32];
        tmem_ld32(src + cb * 64, v[0]);
        tmem_ld32(src + cb * 64 + 32, v[1]);
        tmem_wait_ld();
        reg_fence(v[0]);
        reg_fence(v[1]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {  // 16 columns (two 16-byte chunks) at a time
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[ch / 2][(ch % 2) * 16 + 2 * e]) * mul,
                               __uint_as_float(v[ch / 2][(ch % 2) * 16 + 2 * e + 1]) * mul);
          if (via_tma) {
            const uint32_t rowaddr = stage + cb * C::BLK_BYTES + r * 128;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t chunk = (ch * 2 + u) ^ (r & 7);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowaddr + chunk * 16), "r"(w[4 * u]),
                           "r"(w[4 * u + 1]), "r"(w[4 * u + 2]), "r"(w[4 * u + 3])
                           : "memory");
            }
          } else if (!row_dead) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cb * 64 + ch * 16);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
      if (via_tma) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && kv0 + 32 * wq < sp.seqlen) {
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_store_4d(g == 0 ? &tmDK : &tmDV, stage + kb * C::BLK_BYTES + wq * 4096, kb * 64, sp.h,
                         sp.tma_row0 + kv0 + 32 * wq, sp.tma_b);
          bulk_commit_group();
          bulk_wait_group_read0();  // the stage may be released once the copies have read it
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
                         const CUtensorMap& tdq, const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdParams& p,
                         int max_seqlen, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1) {
  using C = BwdCfg<D>;
  static SmemLimit smem_limit;
  cudaError_t e = smem_limit.ensure(reinterpret_cast<const void*>(fa_bwd_main_kernel<D>), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // The compute warpgroups' setmaxnreg increase is served from the registers
  // the CTA launched with; if the compiler gave the kernel fewer than the
  // split assumes, the increase would never be granted, so refuse to launch.
  static const int launch_regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, fa_bwd_main_kernel<D>) == cudaSuccess ? fa.numRegs : -1;
  }();
  if (launch_regs * C::NUM_THREADS <
      C::NUM_COMPUTE * C::REG_COMPUTE + (C::NUM_THREADS - C::NUM_COMPUTE) * C::REG_OTHER)
    return cudaErrorInvalidConfiguration;
  int sms = 0;
  e = current_sm_count(sms);
  if (e != cudaSuccess) return e;
  BwdParams pm = p;
  pm.sv.npairs = p.nseq * p.sv.H;
  pm.sv.ntiles = (max_seqlen + kTile - 1) / kTile;
  pm.sv.pair_group = pair_group_size(pm.sv.npairs, pm.sv.ntiles, sms);  // one CTA per SM
  const long long ctas = grid_ctas(pm.sv.npairs, pm.sv.ntiles, pm.sv.pair_group);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(ctas));
  const long long pairs = static_cast<long long>(p.rows) * p.sv.H;
  fa_bwd_pre_kernel<D><<<static_cast<unsigned>((pairs * (D / 8) + 255) / 256), 256, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev0 && (e = cudaEventRecord(ev0, s)) != cudaSuccess) return e;
  // The main kernel starts while the pre-pass finishes, and the conversion
  // while the main kernel's last CTAs run (each waits for its predecessor
  // before reading what it wrote).  An event recorded between two kernels
  // (timing the main kernel alone) keeps them apart.
  e = launch_kernel(fa_bwd_main_kernel<D>, grid, dim3(C::NUM_THREADS), C::SMEM_BYTES, s, ev0 == nullptr, tq, tk, tv,
                    tdo, tdq, tdk, tdv, pm);
  if (e != cudaSuccess) return e;
  if (ev1 && (e = cudaEventRecord(ev1, s)) != cudaSuccess) return e;
  const size_t n8 = static_cast<size_t>(pairs) * D / 8;
  return launch_kernel(fa_bwd_post_kernel, dim3(static_cast<unsigned>((n8 + 255) / 256)), dim3(256), 0, s,
                       ev1 == nullptr, p, n8);
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdParams& p, int max_seqlen,
                       cudaStream_t s, cudaEvent_t main_start, cudaEvent_t main_end) {
  if (d == 64) return launch_bwd_d<64>(tq, tk, tv, tdo, tdq, tdk, tdv, p, max_seqlen, s, main_start, main_end);
  return launch_bwd_d<128>(tq, tk, tv, tdo, tdq, tdk, tdv, p, max_seqlen, s, main_start, main_end);
}

}  // namespace fa
