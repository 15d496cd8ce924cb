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
// Each ring stage holds a k-tile of both operands' codes and their scale atoms (A's 128 rows,
// both 128-row bands of B).  Sixteen warps per CTA in four warpgroups (register budgets set
// with setmaxnreg: 56 for the control warps, 152 for the epilogue's):
//   warp 0       TMA producer of the A / B code tiles with the pair form of the copy,
//                completing on the leader's `full` barrier (the leader posts both CTAs' bytes);
//   warp 1       TMEM owner; on the leader, the whole warp issues the pair's MMAs, one elected
//                lane per instruction, once a stage's scales are in TMEM (`sf_ready`);
//   warp 2       TMA producer of the CTA's scale atoms, also in the pair form on the leader's
//                `full` (the leader posts both CTAs' scale bytes);
//   warp 3       on the leader, the whole warp copies each stage's scale atoms of both CTAs
//                from shared memory into the stage's TMEM slot (tcgen05.cp, each CTA's atoms into
//                its own TMEM) and commits to `sf_ready`; issued from a warp of their own, the
//                copies overlap the MMAs on the tensor pipe;
//   warps 4..15  epilogue of the CTA's 128 rows, three warps per TMEM lane quarter (64, 96 and 96
//                of a row's 256 columns); each warp arrives on the leader's `tmem_empty` once
//                per tile (the peer's through a multicast tcgen05.commit).
// The leader's tcgen05.commit is multicast to both CTAs' `empty` and `tmem_full` barriers.
// TMEM: one 256-column accumulator, then one scale slot per ring stage, so a slot is free
// again exactly when its stage is (the producer refills a stage only after the MMAs that read
// its slot have completed).
#pragma once

#include <type_traits>

#include "gemm_kernel.cuh"

namespace bsg {

// KC = k-slabs of 128 bytes of K per ring stage (one wait and one commit per stage).
template <int KIND, int KC>
struct PairCfg {
  static constexpr int BM = 128;  // A rows per CTA (pair tile: 256)
  static constexpr int BN = 256;  // pair tile width; each CTA loads 128 rows of B
  static constexpr int BK_BYTES = 128;
  static constexpr int K_TILE = KC * (KIND == KIND_MX ? 128 : 256);  // elements per stage
  static constexpr int MMA_K = KIND == KIND_MX ? 32 : 64;
  static constexpr int STEPS = K_TILE / MMA_K;                        // 4 MMAs per 128-byte slab
  static constexpr int SF_ATOMS = KC * (KIND == KIND_MX ? 1 : 4);     // per 128-row band per stage
  static constexpr int SLAB_A = BM * BK_BYTES;                        // one 128-byte k-slab of A
  static constexpr int SLAB_B = 128 * BK_BYTES;
  static constexpr int A_BYTES = KC * SLAB_A;
  static constexpr int B_BYTES = KC * SLAB_B;
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
  static constexpr int TMEM_USED = SF_COL0 + STAGES * SF_SLOT_COLS;
  static constexpr int TMEM_COLS = 512;
  // Epilogue: warps 4..15, three per TMEM lane quarter; of a row's 256 columns the first warp of
  // a quarter takes 64, the other two 96 each (TMEM loads of 32 columns, output blocks of 16).
  static constexpr int EPI_WARP0 = 4;
  static constexpr int EPI_WARPS = 12;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 32 * EPI_WARP0 + EPI_THREADS;
  static constexpr int EPI_COLS_FIRST = 64, EPI_COLS = 96;
  static_assert(EPI_COLS_FIRST + 2 * EPI_COLS == BN, "epilogue column split");
  static constexpr int REGS_CTRL = 56, REGS_EPI = 152;
  static_assert(REGS_CTRL + 3 * REGS_EPI <= 512, "register split");
  static_assert(THREADS == 512, "warpgroup layout");
  static constexpr uint32_t IDESC =
      (KIND == KIND_MX ? ((0u << 7) | (0u << 10) | (1u << 23)) : ((1u << 7) | (1u << 10) | (0u << 23))) |
      (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
  static_assert(STAGES >= 2 && STAGES <= 8, "ring");
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory");
};

// Grouped problems never run here (a 256-row pair tile could span two groups); the host plans
// them on 1-SM tiles.
template <int KIND, int KC, int OUT, bool EXT>
__global__ void __launch_bounds__(PairCfg<KIND, KC>::THREADS, 1) bsg_gemm_pair_kernel(const __grid_constant__ PairParams p) {
  using C = PairCfg<KIND, KC>;
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
  // slots: full[0..7], empty[8..15], sf_ready[16..23], tmem_full 32, tmem_empty 33, drain 34,
  // tmem address 35, abort flag 36, copy drain 37.  The leader's `full` completes when both CTAs'
  // code tiles and scale atoms have landed, its `sf_ready` when the stage's scales are in TMEM.
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + 8 + s); };
  auto bar_sf_ready = [&](int s) { return smem_u32(bars + 16 + s); };
  const uint32_t bar_tfull = smem_u32(bars + 32);
  const uint32_t bar_tempty = smem_u32(bars + 33);
  const uint32_t bar_drain = smem_u32(bars + 34);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 35);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 36);
  const uint32_t bar_drain_cp = smem_u32(bars + 37);

  auto stage_a = [&](int s) { return smem0 + s * C::STAGE_BYTES; };
  auto stage_b = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES; };
  auto stage_sfa = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES; };
  auto stage_sfb = [&](int s) { return stage_sfa(s) + C::SFA_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // the leader's code producer (with both CTAs' code bytes) and scale producer (with both
      // CTAs' scale bytes)
      mbar_init(bar_full(s), 2);
      mbar_init(bar_empty(s), 1);     // the leader's multicast commit
      mbar_init(bar_sf_ready(s), 1);  // the leader's copy warp's commit
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, 2 * C::EPI_WARPS);  // one arrival per epilogue warp of each CTA
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain_cp, 1);
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
  // Pointer-agnostic run: the code producer's own copies of the tensor maps, written before the
  // wait (see the 1-SM kernel)
  // (the scale producer likewise for the scale maps, in the next two slots)
  const CUtensorMap* tma = &p.tmap_a;
  const CUtensorMap* tmb = &p.tmap_b;
  const CUtensorMap* tmsa = &p.tmap_sfa;
  const CUtensorMap* tmsb = &p.tmap_sfb;
  if (EXT && p.map_slots != nullptr) {
    CUtensorMap* slot = p.map_slots + MAP_SLOTS_PER_CTA * blockIdx.x;
    // (written by lane 0; every lane of the producer warp acquires them, as the lane that issues
    // its copies is an elected one)
    if (warp == 0 && lane == 0) tmap_remap2(slot, &p.tmap_a, &p.tmap_b, p.remap_a, p.remap_b);
    if (warp == 2 && lane == 0) tmap_remap2(slot + 2, &p.tmap_sfa, &p.tmap_sfb, p.remap_sfa, p.remap_sfb);
    if (warp == 0 || warp == 2) {
      __syncwarp();
      tmap_acquire2(warp == 0 ? slot : slot + 2);
    }
    tma = slot;
    tmb = slot + 1;
    tmsa = slot + 2;
    tmsb = slot + 3;
  }
  griddep_wait();
  griddep_launch_dependents();

  const int pair0 = blockIdx.x >> 1;
  const int pairs = gridDim.x >> 1;

  if (warp < C::EPI_WARP0) {
    setmaxnreg_dec<C::REGS_CTRL>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer (each CTA)
      // The whole warp runs the loop; one elected lane issues each copy.
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool first = true;
      for (int u = pair0; ok && u < p.num_units; u += pairs) {
        const UnitCoord c = decode_unit<EXT>(p, u);
        const int m_blk = c.m_blk * 2 + static_cast<int>(rank & 1u);
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          ok = wait_bounded_cluster_warp(bar_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER);
          if (!ok) break;
          if (first && p.debug_skip_first_load) {
            // test hook: leave this stage unfilled so that the waits downstream run out
          } else {
            // code tiles of both CTAs: one transaction on the leader's barrier
            const uint32_t fb = mapa_shared(bar_full(stage), leader);
            if (is_leader) mbar_arrive_expect_tx_warp(bar_full(stage), 2 * (C::A_BYTES + C::B_BYTES));
#pragma unroll
            for (int j = 0; j < KC; ++j) {  // slabs past K read as zeros (their MMAs are skipped)
              const int x = (kt * KC + j) * C::BK_BYTES;
              const int yb = c.n_blk * C::BN + static_cast<int>(rank & 1u) * 128;
              if (EXT && p.batches > 1)
                tma_load_3d_pair_warp(stage_a(stage) + j * C::SLAB_A, tma, fb, x, m_blk * C::BM, c.batch);
              else
                tma_load_2d_pair_warp(stage_a(stage) + j * C::SLAB_A, tma, fb, x, m_blk * C::BM);
              if (EXT && p.b_entries > 1)
                tma_load_3d_pair_warp(stage_b(stage) + j * C::SLAB_B, tmb, fb, x, yb, c.bsel);
              else
                tma_load_2d_pair_warp(stage_b(stage) + j * C::SLAB_B, tmb, fb, x, yb);
            }
          }
          first = false;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else if (warp == 2) {
      // ---------------------------------------------------------- TMA producer: scale atoms
      // This CTA's scale atoms of the stage, in the pair form of the tiled copy on the leader's
      // `full` (the whole warp runs the loop, one elected lane issues).  Whole boxes always (atoms
      // past the buffer read as zeros), so the byte count is fixed: A's band of this CTA and both
      // bands of B, for each CTA.
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool first = true;
      for (int u = pair0; ok && u < p.num_units; u += pairs) {
        const UnitCoord c = decode_unit<EXT>(p, u);
        const int m_blk = c.m_blk * 2 + static_cast<int>(rank & 1u);
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          ok = wait_bounded_cluster_warp(bar_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER);
          if (!ok) break;
          if (first && p.debug_skip_first_load) {
            // test hook (see the code producer)
          } else {
            const uint32_t fb = mapa_shared(bar_full(stage), leader);
            if (is_leader) mbar_arrive_expect_tx_warp(bar_full(stage), 2 * (C::SFA_BYTES + C::SFB_BYTES));
            const int row = kt * C::SF_ATOMS;
            const int ya = m_blk * p.sfa_atoms_per_band + row;
            if (EXT && p.batches > 1)
              tma_load_3d_pair_warp(stage_sfa(stage), tmsa, fb, 0, ya, c.batch);
            else
              tma_load_2d_pair_warp(stage_sfa(stage), tmsa, fb, 0, ya);
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
              const int yb = (c.n_blk * 2 + rb) * p.sfb_atoms_per_band + row;
              if (EXT && p.b_entries > 1)
                tma_load_3d_pair_warp(stage_sfb(stage) + rb * C::SF_ATOMS * 512, tmsb, fb, 0, yb, c.bsel);
              else
                tma_load_2d_pair_warp(stage_sfb(stage) + rb * C::SF_ATOMS * 512, tmsb, fb, 0, yb);
            }
          }
          first = false;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else if (is_leader) {
      // ---------------------------------------------------------- leader: scale copies (warp 3)
      // and MMAs (warp 1).  Each whole warp runs its loop with warp-uniform values and one
      // elected lane issues each tensor-core instruction.
      const uint32_t tb = __shfl_sync(0xffffffffu, tmem_base, 0);
      const uint32_t s0 = __shfl_sync(0xffffffffu, smem0, 0);
      // descriptors of stage 0; a stage's are these plus its byte offset / 16 (the 14-bit address
      // field holds every shared-memory address, so the sum never carries out of it)
      const uint64_t d_a0 = sdesc_kmajor_sw128(s0);
      const uint64_t d_b0 = sdesc_kmajor_sw128(s0 + C::A_BYTES);
      const uint64_t d_sfa0 = sdesc_sf_atom(s0 + C::A_BYTES + C::B_BYTES);
      const uint64_t d_sfb0 = sdesc_sf_atom(s0 + C::A_BYTES + C::B_BYTES + C::SFA_BYTES);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      if (warp == 3) {
        // scale copies: atom t of A into columns 4t..4t+3 of the stage's slot (lane i of every
        // quarter gets atom row i; the MMA reads, in quarter q, column 4t + q), atom t of B's band
        // b into columns 8t + 4b ..; the atoms K no longer covers are copied too (their MMAs
        // are skipped)
        for (int u = pair0; ok && u < p.num_units; u += pairs) {
          const UnitCoord c = decode_unit<EXT>(p, u);
          for (int kt = c.kt0; kt < c.kt1; ++kt) {
            ok = wait_bounded_cluster_warp(bar_full(stage), phase, abort_flag, p, ST_TIMEOUT_SCALES);
            if (!ok) break;
            tc_fence_after();
            const uint64_t so = static_cast<uint64_t>((stage * C::STAGE_BYTES) >> 4);
            const uint32_t sfa_t = tb + C::SF_COL0 + stage * C::SF_SLOT_COLS;
            const uint32_t sfb_t = sfa_t + C::SFA_COLS;
#pragma unroll
            for (int t = 0; t < C::SF_ATOMS; ++t) {
              tc_cp_sf_atom_pair_warp(sfa_t + 4 * t, d_sfa0 + so + 32 * t);
              tc_cp_sf_atom_pair_warp(sfb_t + 8 * t, d_sfb0 + so + 32 * t);
              tc_cp_sf_atom_pair_warp(sfb_t + 8 * t + 4, d_sfb0 + so + 32 * (C::SF_ATOMS + t));
            }
            tc_commit_pair_mc_warp(bar_sf_ready(stage), static_cast<uint16_t>(1u << rank));
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) {
          // no copy may still be writing TMEM when the CTA frees it
          tc_commit_pair_mc_warp(bar_drain_cp, static_cast<uint16_t>(1u << rank));
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar_drain_cp, 0)) {
              if (globaltimer_ns() - t0 > 10000000ull) {
                atomicOr(p.status, ST_TIMEOUT_DRAIN);
                break;
              }
            }
          }
          __syncwarp();
        }
      } else if (warp == 1) {
        // MMAs: MMA j reads 32 bytes of K at offset 32 (j % 4) of slab j / 4; its scales are in
        // atom j / 4 (MXFP8, byte j % 4 of each word) or atom j (NVFP4)
        uint32_t acc_phase = 0;
        for (int u = pair0; ok && u < p.num_units; u += pairs) {
          const UnitCoord c = decode_unit<EXT>(p, u);
          ok = wait_bounded_cluster_warp(bar_tempty, acc_phase ^ 1u, abort_flag, p, ST_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
          for (int kt = c.kt0; kt < c.kt1; ++kt) {
            // the stage's scales are in TMEM (`sf_ready`), which the copy warp commits only after
            // it saw the stage's `full` (codes and scale atoms landed) and its copies completed;
            // waiting on `full` here as well cost ~5 us at 8192^3
            ok = wait_bounded_cluster_warp(bar_sf_ready(stage), phase, abort_flag, p, ST_TIMEOUT_MMA);
            if (!ok) break;
            tc_fence_after();
            const int steps = min(C::STEPS, (p.K - kt * C::K_TILE + C::MMA_K - 1) / C::MMA_K);
            const uint64_t so = static_cast<uint64_t>((stage * C::STAGE_BYTES) >> 4);
            const uint32_t sfa_t = tb + C::SF_COL0 + stage * C::SF_SLOT_COLS;
            const uint32_t sfb_t = sfa_t + C::SFA_COLS;
            const uint32_t acc0 = kt > c.kt0 ? 1u : 0u;
            auto mma = [&](int j, uint32_t acc) {
              const uint32_t jj = static_cast<uint32_t>(j & 3), slab = static_cast<uint32_t>(j >> 2);
              const uint64_t ad = d_a0 + so + ((slab * C::SLAB_A + 32 * jj) >> 4);
              const uint64_t bd = d_b0 + so + ((slab * C::SLAB_B + 32 * jj) >> 4);
              if constexpr (KIND == KIND_MX)
                tc_mma_mxf8_pair_warp(tb, ad, bd, C::IDESC | (jj << 4) | (jj << 29), sfa_t + 4 * slab,
                                      sfb_t + 8 * slab, acc);
              else
                tc_mma_nvf4_pair_warp(tb, ad, bd, C::IDESC, sfa_t + 4 * j, sfb_t + 8 * j, acc);
            };
            if (steps == C::STEPS) {
#pragma unroll
              for (int j = 0; j < C::STEPS; ++j) mma(j, j == 0 ? acc0 : 1u);  // straight-line issue
            } else {
              for (int j = 0; j < steps; ++j) mma(j, j == 0 ? acc0 : 1u);  // the last, partial k-tile
            }
            tc_commit_pair_mc_warp(bar_empty(stage), pair_mask);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair_mc_warp(bar_tfull, pair_mask);
          acc_phase ^= 1u;
        }
        if (!ok) {
          tc_commit_pair_mc_warp(bar_drain, static_cast<uint16_t>(1u << rank));
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar_drain, 0)) {
              if (globaltimer_ns() - t0 > 10000000ull) {
                atomicOr(p.status, ST_TIMEOUT_DRAIN);
                break;
              }
            }
          }
          __syncwarp();
        }
      }
    }
  } else {
    setmaxnreg_inc<C::REGS_EPI>();
    // ------------------------------------------------------------ epilogue (each CTA, 12 warps)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int part = (warp - C::EPI_WARP0) >> 2;  // 0: columns 0..63, 1: 64..159, 2: 160..255
    const int col0 = part == 0 ? 0 : C::EPI_COLS_FIRST + (part - 1) * C::EPI_COLS;
    const float alpha0 = (p.flags & F_ALPHA_DEVICE) ? __ldg(p.alpha_dev) : p.alpha;
    const uint16_t leader_mask = static_cast<uint16_t>(1u << leader);
    uint32_t acc_phase = 0;
    // The whole row segment comes out of TMEM before any arithmetic and the accumulator is
    // released at once: the next tile's MMAs need all of it, and holding it through the epilogue
    // math stalled them for longer than the math itself takes (the NVFP4 output too: holding
    // the only accumulator through its encoding, 8192^3 took 315 us against 180 us with a 16-bit
    // output).
    auto tile = [&](auto cols_tag) {
      constexpr int COLS = decltype(cols_tag)::value;
      for (int u = pair0; u < p.num_units; u += pairs) {
        const UnitCoord c = decode_unit<EXT>(p, u);
        const float alpha = unit_alpha<EXT>(p, c, alpha0);
        // each warp on its own: a warp that gives up leaves the loop, and none waits for another
        if (!wait_bounded_cluster(bar_tfull, acc_phase, abort_flag, p, ST_TIMEOUT_EPILOGUE)) break;
        tc_fence_after();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const int m = (c.m_blk * 2 + static_cast<int>(rank & 1u)) * C::BM + row;
        const int nbase = c.n_blk * C::BN;
        uint32_t r[COLS];
#pragma unroll
        for (int ch = 0; ch < COLS / 32; ++ch)
          tmem_ld_32x32b_x32(t_row + col0 + ch * 32, reinterpret_cast<uint32_t(&)[32]>(r[32 * ch]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (is_leader)
            mbar_arrive(bar_tempty);
          else
            tc_commit_pair_mc(bar_tempty, leader_mask);
        }
        epilogue_row<OUT, COLS / 16, EXT>(p, c.batch, m, m < p.M, nbase + col0, r, alpha);
        acc_phase ^= 1u;
      }
    };
    if (part == 0)
      tile(std::integral_constant<int, C::EPI_COLS_FIRST>{});
    else
      tile(std::integral_constant<int, C::EPI_COLS>{});
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

template <int KIND, int KC, int OUT, bool EXT = false>
bool fill_pair_kernel_info(GemmKernelInfo* info) {
  using C = PairCfg<KIND, KC>;
  info->fn = reinterpret_cast<const void*>(&bsg_gemm_pair_kernel<KIND, KC, OUT, EXT>);
  info->kc = KC;
  info->smem_bytes = C::SMEM_BYTES;
  info->threads = C::THREADS;
  info->bn = C::BN;
  info->stages = C::STAGES;
  info->stage_bytes = C::STAGE_BYTES;
  return true;
}

}  // namespace bsg
