// CTA-pair block-scaled GEMM kernel for sm_103a (tcgen05 cta_group::2).
//
// Two CTAs of a 2-CTA cluster compute one 256 x 256 output tile with M = 256 MMAs issued by
// the even CTA (the leader): each CTA loads 128 rows of A and 128 of the tile's 256 rows of B
// into its own shared memory, and its TMEM receives its 128 rows of the accumulator.  Per SM,
// the shared-memory traffic per MMA is two thirds of the 1-SM 128 x 256 tile's, which is what
// limits the 1-SM kernel on large problems.  This is the 2-SM schedule of the pages
// ("[QST] Performance overhead ...": KernelConfigM256 / KernelConfigDefault with
// KernelTmaWarpSpecialized2SmNvf4Sm100; "Add Cutlass MxFp8 Block Scale Matrix
// Multiplication": MmaTileShape 256 x 256 x 256 over a cluster, PerSmTileShape 128 x 256).
//
// Warps (both CTAs): 0 TMA producer, 1 TMEM owner / MMA issuer (the leader's lane 0 issues
// the pair's scale copies and MMAs), 2..9 epilogue.
// Synchronisation without per-stage thread handshakes between the CTAs: both CTAs' TMA loads
// of a stage complete on the leader's `full` barrier (the leader posts the byte count of both);
// the leader's tcgen05.commit is multicast to both CTAs' `empty` and `tmem_full` barriers; the
// scale atoms go to each CTA's own TMEM through pairwise tcgen05.cp (each CTA holds A's and
// both of B's 128-row scale bands in its own shared memory); each epilogue warp arrives on the
// leader's `tmem_empty` once per tile.
#pragma once

#include "gemm_kernel.cuh"

namespace bsg {

template <int KIND>
struct PairCfg {
  static constexpr int BM = 128;  // A rows per CTA (pair tile: 256)
  static constexpr int BN = 256;  // pair tile width; each CTA loads 128 rows of B
  static constexpr int BK_BYTES = 128;
  static constexpr int K_TILE = KIND == KIND_MX ? 128 : 256;
  static constexpr int MMA_K = KIND == KIND_MX ? 32 : 64;
  static constexpr int STEPS = K_TILE / MMA_K;
  static constexpr int SF_ATOMS = KIND == KIND_MX ? 1 : 4;
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = 128 * BK_BYTES;
  static constexpr int SFA_BYTES = SF_ATOMS * 512;
  static constexpr int SFB_BYTES = 2 * SF_ATOMS * 512;  // both 128-row bands of the tile's B
  static constexpr int STAGE_RAW = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int AUX_BYTES = 1024;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - AUX_BYTES - 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + AUX_BYTES + 1024;
  static constexpr int SFA_COLS = 4 * SF_ATOMS;  // per scale slot: A's 128 rows
  static constexpr int SFB_COLS = 8 * SF_ATOMS;  // B's 256 rows
  static constexpr int SF_SLOT_COLS = SFA_COLS + SFB_COLS;
  static constexpr int SF_COL0 = BN;             // one 256-column accumulator first
  static constexpr int TMEM_USED = SF_COL0 + 2 * SF_SLOT_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int EPI_WARP0 = 2;
  static constexpr int THREADS = 32 * EPI_WARP0 + EPI_THREADS;
  static constexpr uint32_t IDESC =
      (KIND == KIND_MX ? ((0u << 7) | (0u << 10) | (1u << 23)) : ((1u << 7) | (1u << 10) | (0u << 23))) |
      (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
  static_assert(STAGES >= 2 && STAGES <= 8, "ring");
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory");
};

template <int KIND, int OUT>
__global__ void __launch_bounds__(PairCfg<KIND>::THREADS, 1) bsg_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  using C = PairCfg<KIND>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
  const uint32_t smem0 = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // even: leader, odd: peer
  const uint32_t leader = rank & ~1u;
  const bool is_leader = (rank & 1u) == 0;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << leader);

  uint8_t* aux = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  // slots: full[0..7], empty[8..15], tmem_full 16, tmem_empty 17, drain 18
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + 8 + s); };
  const uint32_t bar_tfull = smem_u32(bars + 16);
  const uint32_t bar_tempty = smem_u32(bars + 17);
  const uint32_t bar_drain = smem_u32(bars + 18);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 20);

  auto stage_a = [&](int s) { return smem0 + s * C::STAGE_BYTES; };
  auto stage_b = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES; };
  auto stage_sfa = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES; };
  auto stage_sfb = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES + C::SFA_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full(s), 1);   // the leader's producer arrives (with both CTAs' bytes)
      mbar_init(bar_empty(s), 1);  // the leader's multicast commit
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, 2 * C::EPI_WARPS);  // one arrival per epilogue warp of each CTA
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
    prefetch_tmap(&p.tmap_sfa);
    prefetch_tmap(&p.tmap_sfb);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();
  griddep_launch_dependents();

  const int pair0 = blockIdx.x >> 1;
  const int pairs = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (each CTA)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool first = true;
      for (int u = pair0; ok && u < p.num_units; u += pairs) {
        const UnitCoord c = decode_unit(p, u);
        const int m_blk = c.m_blk * 2 + static_cast<int>(rank & 1u);
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!wait_bounded_cluster(bar_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          // The pair's stage is one transaction on the leader's barrier: A, B and the scale
          // atoms of both CTAs, whole boxes (bands past the scale buffers read as zeros).
          const uint32_t fb = mapa_shared(bar_full(stage), leader);
          if (first && p.debug_skip_first_load) {
            // test hook: leave this stage unfilled so that the waits downstream run out
          } else {
            if (is_leader) mbar_arrive_expect_tx(bar_full(stage), 2 * C::STAGE_RAW);
            tma_load_2d_pair(stage_a(stage), &p.tmap_a, fb, kt * C::BK_BYTES, m_blk * C::BM);
            tma_load_2d_pair(stage_b(stage), &p.tmap_b, fb, kt * C::BK_BYTES,
                             c.n_blk * C::BN + static_cast<int>(rank & 1u) * 128);
            tma_load_2d_pair(stage_sfa(stage), &p.tmap_sfa, fb, 0,
                             (m_blk * p.sfa_atoms_per_band + kt * C::SF_ATOMS) * 4);
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
              tma_load_2d_pair(stage_sfb(stage) + rb * C::SF_ATOMS * 512, &p.tmap_sfb, fb, 0,
                               ((c.n_blk * 2 + rb) * p.sfb_atoms_per_band + kt * C::SF_ATOMS) * 4);
          }
          first = false;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader, lane 0)
    if (is_leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      bool ok = true;
      for (int u = pair0; ok && u < p.num_units; u += pairs) {
        const UnitCoord c = decode_unit(p, u);
        if (!wait_bounded_cluster(bar_tempty, acc_phase ^ 1u, abort_flag, p, ST_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!wait_bounded(bar_full(stage), phase, abort_flag, p, ST_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int k_rem = p.K - kt * C::K_TILE;
          const int steps = min(C::STEPS, (k_rem + C::MMA_K - 1) / C::MMA_K);
          const uint32_t sfa_t = tmem_base + C::SF_COL0 + slot * C::SF_SLOT_COLS;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
          const uint32_t sa = stage_a(stage), sb = stage_b(stage);
          const uint32_t ssfa = stage_sfa(stage), ssfb = stage_sfb(stage);
          if constexpr (KIND == KIND_MX) {
            tc_cp_sf_atom_pair(sfa_t, sdesc_sf_atom(ssfa));
            tc_cp_sf_atom_pair(sfb_t, sdesc_sf_atom(ssfb));
            tc_cp_sf_atom_pair(sfb_t + 4, sdesc_sf_atom(ssfb + 512));
            for (int j = 0; j < steps; ++j) {
              const uint32_t idesc = C::IDESC | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
              tc_mma_mxf8_pair(tmem_base, sdesc_kmajor_sw128(sa + 32 * j), sdesc_kmajor_sw128(sb + 32 * j), idesc,
                               sfa_t, sfb_t, (kt > c.kt0 || j > 0) ? 1u : 0u);
            }
          } else {
            for (int j = 0; j < steps; ++j) {
              tc_cp_sf_atom_pair(sfa_t + 4 * j, sdesc_sf_atom(ssfa + 512 * j));
              tc_cp_sf_atom_pair(sfb_t + 8 * j, sdesc_sf_atom(ssfb + 512 * j));
              tc_cp_sf_atom_pair(sfb_t + 8 * j + 4, sdesc_sf_atom(ssfb + C::SF_ATOMS * 512 + 512 * j));
            }
            for (int j = 0; j < steps; ++j)
              tc_mma_nvf4_pair(tmem_base, sdesc_kmajor_sw128(sa + 32 * j), sdesc_kmajor_sw128(sb + 32 * j), C::IDESC,
                               sfa_t + 4 * j, sfb_t + 8 * j, (kt > c.kt0 || j > 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(bar_empty(stage), pair_mask);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          slot ^= 1;
        }
        if (!ok) break;
        tc_commit_pair_mc(bar_tfull, pair_mask);
        acc_phase ^= 1u;
      }
      if (!ok) {
        tc_commit_pair_mc(bar_drain, static_cast<uint16_t>(1u << rank));
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_drain, 0)) {
          if (globaltimer_ns() - t0 > 10000000ull) {
            atomicOr(p.status, ST_TIMEOUT_DRAIN);
            break;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (each CTA, 8 warps)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    constexpr int HC = C::BN / 2;
    const int col0 = ((warp - C::EPI_WARP0) >> 2) * HC;
    const float alpha = (p.flags & F_ALPHA_DEVICE) ? __ldg(p.alpha_dev) : p.alpha;
    const uint32_t leader_tempty = mapa_shared(bar_tempty, leader);
    uint32_t acc_phase = 0;
    for (int u = pair0; u < p.num_units; u += pairs) {
      const UnitCoord c = decode_unit(p, u);
      bool ok = wait_bounded_cluster(bar_tfull, acc_phase, abort_flag, p, ST_TIMEOUT_EPILOGUE);
      ok = named_bar_and(1, C::EPI_THREADS, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int m = (c.m_blk * 2 + static_cast<int>(rank & 1u)) * C::BM + row;
      const int nbase = c.n_blk * C::BN;
      uint32_t packed[HC / 2];
#pragma unroll
      for (int ch = 0; ch < HC / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + col0 + ch * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[8 * g + i]);
          epi_pack<OUT, 8>(p, nbase + col0 + ch * 32 + 8 * g, v, alpha, &packed[ch * 16 + 4 * g]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(leader_tempty);
      if (m < p.M) {
        uint16_t* drow = static_cast<uint16_t*>(p.d) + static_cast<size_t>(m) * p.N;
#pragma unroll
        for (int g = 0; g < HC / 8; ++g) {
          const int n = nbase + col0 + 8 * g;
          if (n < p.N)
            *reinterpret_cast<uint4*>(drow + n) =
                make_uint4(packed[4 * g], packed[4 * g + 1], packed[4 * g + 2], packed[4 * g + 3]);
        }
      }
      acc_phase ^= 1u;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees TMEM or leaves while the pair's MMAs may use its memory
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int KIND, int OUT>
bool fill_pair_kernel_info(GemmKernelInfo* info) {
  using C = PairCfg<KIND>;
  info->fn = reinterpret_cast<const void*>(&bsg_gemm_pair_kernel<KIND, OUT>);
  info->smem_bytes = C::SMEM_BYTES;
  info->threads = C::THREADS;
  info->bn = C::BN;
  info->stages = C::STAGES;
  return true;
}

}  // namespace bsg
