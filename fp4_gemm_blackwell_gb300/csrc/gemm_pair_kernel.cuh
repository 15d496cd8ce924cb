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
// Sixteen warps per CTA in four warpgroups (register budgets set with setmaxnreg):
//   warp 0       TMA producer of the A / B code tiles with the pair form of the copy,
//                completing on the leader's `full` barrier (the leader posts both CTAs' bytes);
//   warp 1       TMEM owner; the leader's lane 0 issues the pair's MMAs;
//   warp 2       TMA producer of the CTA's scale atoms (A's 128 rows, both 128-row bands of
//                B), completing on its own `sf_full` barrier;
//   warps 4..7   scale warps: copy each stage's scale atoms into the CTA's own TMEM slot
//                (tcgen05.st) and arrive on the leader's `full` barrier (the peer's through a
//                multicast tcgen05.commit);
//   warps 8..15  epilogue of the CTA's 128 rows; each warp arrives on the leader's
//                `tmem_empty` once per tile (the peer's through a multicast tcgen05.commit).
// The leader's tcgen05.commit is multicast to both CTAs' `empty` and `tmem_full` barriers.
#pragma once

#include "gemm_kernel.cuh"

namespace bsg {

// KC = k-tiles of 128 bytes of K per ring stage (one wait and one commit per stage).
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
  // SEP: the scale atoms have their own two-stage ring and two TMEM slots, apart from the code
  // ring (NVFP4 with two k-slabs: 12 KB of atoms per stage would leave room for only two 76 KB
  // stages, and 96 TMEM columns per slot for only two slots).  The scale warps release a scale
  // stage once they have copied it; a TMEM slot is free again once the MMAs of the code stage
  // that last used it have completed (that code stage's `empty` barrier).
  static constexpr bool SEP = KIND == KIND_NV && KC == 2;
  static constexpr int SF_STAGE_BYTES = (SFA_BYTES + SFB_BYTES + 1023) / 1024 * 1024;
  static constexpr int SF_STAGES = SEP ? 2 : 0;
  static constexpr int STAGE_RAW = A_BYTES + B_BYTES + (SEP ? 0 : SFA_BYTES + SFB_BYTES);
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int AUX_BYTES = 1024;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - AUX_BYTES - 1024 - SF_STAGES * SF_STAGE_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + SF_STAGES * SF_STAGE_BYTES + AUX_BYTES + 1024;
  static constexpr int SFA_COLS = 4 * SF_ATOMS;  // per scale slot: A's 128 rows
  static constexpr int SFB_COLS = 8 * SF_ATOMS;  // B's 256 rows
  static constexpr int SF_SLOT_COLS = SFA_COLS + SFB_COLS;
  static constexpr int SF_COL0 = BN;             // one 256-column accumulator first
  static constexpr int SF_SLOTS = SEP ? SF_STAGES : STAGES;
  static constexpr int TMEM_USED = SF_COL0 + SF_SLOTS * SF_SLOT_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int SCALE_WARP0 = 4;
  static constexpr int EPI_WARP0 = 8;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 32 * EPI_WARP0 + EPI_THREADS;
  static constexpr int REGS_CTRL = 56, REGS_SCALE = 80, REGS_EPI = 184;
  static_assert(REGS_CTRL + REGS_SCALE + 2 * REGS_EPI <= 512, "register split");
  static_assert(THREADS == 512, "warpgroup layout");
  static constexpr uint32_t IDESC =
      (KIND == KIND_MX ? ((0u << 7) | (0u << 10) | (1u << 23)) : ((1u << 7) | (1u << 10) | (0u << 23))) |
      (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
  static_assert(STAGES >= 2 && STAGES <= 8, "ring");
  static_assert(SF_ATOMS <= 4 || SF_ATOMS % 4 == 0, "scale-warp stores");
  static_assert(TMEM_USED <= TMEM_COLS, "tensor memory");
};

// Grouped problems never run here (a 256-row pair tile could span two groups); the host plans
// them on 1-SM tiles.
template <int KIND, int KC, int OUT, bool EXT>
__global__ void __launch_bounds__(PairCfg<KIND, KC>::THREADS, 1) bsg_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
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

  const uint32_t sf0 = smem0 + C::STAGES * C::STAGE_BYTES;  // separate scale ring (SEP)
  uint8_t* aux = smem + C::STAGES * C::STAGE_BYTES + C::SF_STAGES * C::SF_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  // slots: full[0..7], empty[8..15], sf_full[16..23], tmem_full 32, tmem_empty 33, drain 34,
  // tmem address 35, abort flag 36; with a separate scale ring also sf_empty[40..47].  The
  // leader's `full` completes when both CTAs' code tiles have landed and both CTAs' scale warps
  // have filled their TMEM slots: one wait per stage for the MMA issuer.
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + 8 + s); };
  auto bar_sf_full = [&](int s) { return smem_u32(bars + 16 + s); };
  auto bar_sf_empty = [&](int t) { return smem_u32(bars + 40 + t); };  // scale stage copied (SEP)
  const uint32_t bar_tfull = smem_u32(bars + 32);
  const uint32_t bar_tempty = smem_u32(bars + 33);
  const uint32_t bar_drain = smem_u32(bars + 34);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 35);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 36);

  auto stage_a = [&](int s) { return smem0 + s * C::STAGE_BYTES; };
  auto stage_b = [&](int s) { return smem0 + s * C::STAGE_BYTES + C::A_BYTES; };
  // scale atoms of stage s (SEP: of scale stage s)
  auto stage_sfa = [&](int s) {
    return C::SEP ? sf0 + s * C::SF_STAGE_BYTES : smem0 + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
  };
  auto stage_sfb = [&](int s) { return stage_sfa(s) + C::SFA_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // the leader's producer (with both CTAs' code bytes) and, without a separate scale ring,
      // the scale warps of both CTAs
      mbar_init(bar_full(s), 1 + 8);
      mbar_init(bar_empty(s), 1);    // the leader's multicast commit
      mbar_init(bar_sf_full(s), 1);  // this CTA's producer (scale bytes)
    }
    for (int t = 0; t < C::SF_STAGES; ++t) mbar_init(bar_sf_empty(t), 4);  // this CTA's scale warps
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, 2 * C::EPI_WARPS);  // one arrival per epilogue warp of each CTA
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
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
  const CUtensorMap* tma = &p.tmap_a;
  const CUtensorMap* tmb = &p.tmap_b;
  if (EXT && p.map_slots != nullptr) {
    CUtensorMap* slot = p.map_slots + 2 * blockIdx.x;
    if (warp == 0 && lane == 0) {
      tmap_remap2(slot, &p.tmap_a, &p.tmap_b, p.remap_a, p.remap_b);
    }
    tma = slot;
    tmb = slot + 1;
  }
  griddep_wait();
  griddep_launch_dependents();

  const int pair0 = blockIdx.x >> 1;
  const int pairs = gridDim.x >> 1;

  if (warp < C::SCALE_WARP0) {
    setmaxnreg_dec<C::REGS_CTRL>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer (each CTA)
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        bool first = true;
        for (int u = pair0; ok && u < p.num_units; u += pairs) {
          const UnitCoord c = decode_unit<EXT>(p, u);
          const int m_blk = c.m_blk * 2 + static_cast<int>(rank & 1u);
          for (int kt = c.kt0; kt < c.kt1; ++kt) {
            if (!wait_bounded_cluster(bar_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER)) {
              ok = false;
              break;
            }
            if (first && p.debug_skip_first_load) {
              // test hook: leave this stage unfilled so that the waits downstream run out
            } else {
              // code tiles of both CTAs: one transaction on the leader's barrier
              const uint32_t fb = mapa_shared(bar_full(stage), leader);
              if (is_leader) mbar_arrive_expect_tx(bar_full(stage), 2 * (C::A_BYTES + C::B_BYTES));
#pragma unroll
              for (int j = 0; j < KC; ++j) {  // slabs past K read as zeros (their MMAs are skipped)
                const int x = (kt * KC + j) * C::BK_BYTES;
                const int yb = c.n_blk * C::BN + static_cast<int>(rank & 1u) * 128;
                if (EXT && p.batches > 1)
                  tma_load_3d_pair(stage_a(stage) + j * C::SLAB_A, tma, fb, x, m_blk * C::BM, c.batch);
                else
                  tma_load_2d_pair(stage_a(stage) + j * C::SLAB_A, tma, fb, x, m_blk * C::BM);
                if (EXT && p.b_entries > 1)
                  tma_load_3d_pair(stage_b(stage) + j * C::SLAB_B, tmb, fb, x, yb, c.bsel);
                else
                  tma_load_2d_pair(stage_b(stage) + j * C::SLAB_B, tmb, fb, x, yb);
              }
            }
            first = false;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    } else if (warp == 2) {
      // ---------------------------------------------------------- TMA producer: scale atoms
      // A second issuing thread (each copy instruction holds its thread for a hundred-odd
      // cycles): this CTA's scale atoms, on its own barrier; into the code ring's stages, or
      // (SEP) into the scale ring, refilled once the scale warps have copied a stage.
      constexpr int NR = C::SEP ? C::SF_STAGES : C::STAGES;
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        bool first = true;
        for (int u = pair0; ok && u < p.num_units; u += pairs) {
          const UnitCoord c = decode_unit<EXT>(p, u);
          const int m_blk = c.m_blk * 2 + static_cast<int>(rank & 1u);
          const bool a_band = m_blk < p.sfa_bands;  // false for the pair's second m-tile past M
          int bands = 0;
#pragma unroll
          for (int rb = 0; rb < 2; ++rb) bands += (c.n_blk * 2 + rb < p.sfb_bands) ? 1 : 0;
          for (int kt = c.kt0; kt < c.kt1; ++kt) {
            const bool free_ = C::SEP ? wait_bounded(bar_sf_empty(stage), phase ^ 1u, abort_flag, p, ST_TIMEOUT_PRODUCER)
                                      : wait_bounded_cluster(bar_empty(stage), phase ^ 1u, abort_flag, p,
                                                             ST_TIMEOUT_PRODUCER);
            if (!free_) {
              ok = false;
              break;
            }
            const int k_rem = p.K - kt * C::K_TILE;
            const int steps = min(C::STEPS, (k_rem + C::MMA_K - 1) / C::MMA_K);
            const int sf_atoms = KIND == KIND_MX ? (steps + 3) / 4 : steps;  // atoms K still covers
            if (first && p.debug_skip_first_load) {
              // test hook (see the code producer)
            } else {
              const uint32_t sb = bar_sf_full(stage);
              mbar_arrive_expect_tx(sb, static_cast<uint32_t>(((a_band ? 1 : 0) + bands) * sf_atoms * 512));
              if (a_band)
                bulk_load(stage_sfa(stage),
                          p.sfa + c.batch * p.sfa_batch + (static_cast<size_t>(m_blk) * p.sfa_atoms_per_band +
                                   static_cast<size_t>(kt) * C::SF_ATOMS) * 512,
                          sf_atoms * 512, sb);
#pragma unroll
              for (int rb = 0; rb < 2; ++rb) {
                const int band = c.n_blk * 2 + rb;
                if (band < p.sfb_bands)
                  bulk_load(stage_sfb(stage) + rb * C::SF_ATOMS * 512,
                            p.sfb + c.bsel * p.sfb_batch + (static_cast<size_t>(band) * p.sfb_atoms_per_band +
                                     static_cast<size_t>(kt) * C::SF_ATOMS) * 512,
                            sf_atoms * 512, sb);
              }
            }
            first = false;
            if (++stage == NR) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (leader, lane 0)
      if (is_leader && lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int sst = 0;  // TMEM scale slot (SEP): the scale ring's stage
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int u = pair0; ok && u < p.num_units; u += pairs) {
          const UnitCoord c = decode_unit<EXT>(p, u);
          if (!wait_bounded_cluster(bar_tempty, acc_phase ^ 1u, abort_flag, p, ST_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kt = c.kt0; kt < c.kt1; ++kt) {
            if (!wait_bounded_cluster(bar_full(stage), phase, abort_flag, p, ST_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int k_rem = p.K - kt * C::K_TILE;
            const int steps = min(C::STEPS, (k_rem + C::MMA_K - 1) / C::MMA_K);
            // the scale warps of both CTAs have put this stage's scales in their TMEM slots
            const uint32_t sfa_t = tmem_base + C::SF_COL0 + (C::SEP ? sst : stage) * C::SF_SLOT_COLS;
            const uint32_t sfb_t = sfa_t + C::SFA_COLS;
            const uint32_t sa = stage_a(stage), sb = stage_b(stage);
            // MMA j reads 32 bytes of K at offset 32 (j % 4) of slab j / 4; its scales are in atom
            // j / 4 (MXFP8, byte j % 4 of each word) or atom j (NVFP4)
            if constexpr (KIND == KIND_MX) {
              for (int j = 0; j < steps; ++j) {
                const uint32_t jj = static_cast<uint32_t>(j & 3), slab = static_cast<uint32_t>(j >> 2);
                const uint32_t idesc = C::IDESC | (jj << 4) | (jj << 29);
                tc_mma_mxf8_pair(tmem_base, sdesc_kmajor_sw128(sa + slab * C::SLAB_A + 32 * jj),
                                 sdesc_kmajor_sw128(sb + slab * C::SLAB_B + 32 * jj), idesc, sfa_t + 4 * slab,
                                 sfb_t + 8 * slab, (kt > c.kt0 || j > 0) ? 1u : 0u);
              }
            } else {
              for (int j = 0; j < steps; ++j) {
                const uint32_t jj = static_cast<uint32_t>(j & 3), slab = static_cast<uint32_t>(j >> 2);
                tc_mma_nvf4_pair(tmem_base, sdesc_kmajor_sw128(sa + slab * C::SLAB_A + 32 * jj),
                                 sdesc_kmajor_sw128(sb + slab * C::SLAB_B + 32 * jj), C::IDESC, sfa_t + 4 * j,
                                 sfb_t + 8 * j, (kt > c.kt0 || j > 0) ? 1u : 0u);
              }
            }
            tc_commit_pair_mc(bar_empty(stage), pair_mask);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            if constexpr (C::SEP) {
              if (++sst == C::SF_STAGES) sst = 0;
            }
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
    }
  } else if (warp < C::EPI_WARP0) {
    setmaxnreg_dec<C::REGS_SCALE>();
    // ------------------------------------------------------------ scale warps (each CTA)
    // The layout a 32x128b.warpx4 copy of the atoms produces, per stage slot: lane i, column
    // 4t + k holds the four scales of A row 32k + i of atom t (this CTA's 128 rows), and column
    // 8t + 4b + k those of B row 128b + 32k + i (the pair tile's 256 rows).  Of A's four columns
    // the MMA reads, in lane quarter q, only column 4t + q (the scales of its own rows 32q + i),
    // so each scale warp writes only that one: a quarter of A's bytes (measured: results
    // unchanged, NVFP4 8192^3 182.3 -> 179.7 us).
    // With a separate scale ring (SEP) the stage index is the scale stage, which is also the TMEM
    // slot: it is refilled once the MMAs that read its previous contents, those of the ring stage
    // SF_STAGES back, have completed, which the leader's commit to that code stage's `empty`
    // barrier (multicast to both CTAs) tells.  Either way the scale warps arrive on the code
    // stage's `full` barrier, so the MMA issuer waits once per stage and commits once.
    constexpr int NR = C::SEP ? C::SF_STAGES : C::STAGES;
    const int q = warp & 3;
    const uint16_t leader_mask = static_cast<uint16_t>(1u << leader);
    int stage = 0;
    uint32_t phase = 0;
    int cs = 0;                   // code stage of this k-stage (SEP)
    int cs_old = 0, lag = 0;      // code stage SF_STAGES k-stages back, once there is one (SEP)
    uint32_t ph_old = 0;
    bool ok = true;
    for (int u = pair0; ok && u < p.num_units; u += pairs) {
      const UnitCoord c = decode_unit<EXT>(p, u);
      for (int kt = c.kt0; kt < c.kt1; ++kt) {
        ok = __all_sync(0xffffffffu, wait_bounded(bar_sf_full(stage), phase, abort_flag, p, ST_TIMEOUT_SCALES));
        if (!ok) break;
        const uint32_t slot = tmem_base + C::SF_COL0 + stage * C::SF_SLOT_COLS + (static_cast<uint32_t>(q * 32) << 16);
        // atoms in groups of up to four: 16 A columns and 32 B columns per group
        constexpr int NA = C::SF_ATOMS;
        constexpr int GA = NA < 4 ? NA : 4;
        auto load_group = [&](int g0, uint32_t (&a)[GA], uint32_t (&b)[8 * GA]) {
#pragma unroll
          for (int t = 0; t < GA; ++t) {
            a[t] = lds_u32(stage_sfa(stage) + 512 * (g0 + t) + 16 * lane + 4 * q);  // this quarter's word
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
              const uint4 w = lds_u4(stage_sfb(stage) + rb * NA * 512 + 512 * (g0 + t) + 16 * lane);
              b[(2 * t + rb) * 4] = w.x;
              b[(2 * t + rb) * 4 + 1] = w.y;
              b[(2 * t + rb) * 4 + 2] = w.z;
              b[(2 * t + rb) * 4 + 3] = w.w;
            }
          }
        };
        // The first group is read from shared memory before the TMEM slot is known to be free
        // (SEP: the MMAs of the stage SF_STAGES back may still be reading it), so that only the
        // stores into TMEM follow the MMAs' completion.
        uint32_t a[GA], b[8 * GA];
        load_group(0, a, b);
        if constexpr (C::SEP) {
          if (lag == C::SF_STAGES) {
            ok = __all_sync(0xffffffffu,
                            wait_bounded_cluster(bar_empty(cs_old), ph_old, abort_flag, p, ST_TIMEOUT_SCALES));
            if (!ok) break;
            if (++cs_old == C::STAGES) {
              cs_old = 0;
              ph_old ^= 1u;
            }
          } else {
            ++lag;
          }
        }
#pragma unroll
        for (int t = 0; t < GA; ++t) tmem_st_32x32b_x1(slot + 4 * t + q, a[t]);
        tmem_st_cols(slot + C::SFA_COLS, b);
#pragma unroll
        for (int g0 = GA; g0 < NA; g0 += GA) {
          load_group(g0, a, b);
#pragma unroll
          for (int t = 0; t < GA; ++t) tmem_st_32x32b_x1(slot + 4 * (g0 + t) + q, a[t]);
          tmem_st_cols(slot + C::SFA_COLS + 8 * g0, b);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // The peer signals through the tensor-core commit path, which arrives on the leader's
          // barrier without holding this thread for the cluster round trip that a remote
          // mbarrier arrive takes (its stores to TMEM are complete: tcgen05.wait::st above).
          const uint32_t ready = C::SEP ? bar_full(cs) : bar_full(stage);
          if (is_leader)
            mbar_arrive(ready);
          else
            tc_commit_pair_mc(ready, leader_mask);
          if (C::SEP) mbar_arrive(bar_sf_empty(stage));  // the scale stage may be refilled
        }
        if (C::SEP && ++cs == C::STAGES) cs = 0;
        if (++stage == NR) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    setmaxnreg_inc<C::REGS_EPI>();
    // ------------------------------------------------------------ epilogue (each CTA, 8 warps)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    constexpr int HC = C::BN / 2;
    const int col0 = ((warp - C::EPI_WARP0) >> 2) * HC;
    const float alpha0 = (p.flags & F_ALPHA_DEVICE) ? __ldg(p.alpha_dev) : p.alpha;
    const uint16_t leader_mask = static_cast<uint16_t>(1u << leader);
    uint32_t acc_phase = 0;
    for (int u = pair0; u < p.num_units; u += pairs) {
      const UnitCoord c = decode_unit<EXT>(p, u);
      const float alpha = unit_alpha<EXT>(p, c, alpha0);
      bool ok = wait_bounded_cluster(bar_tfull, acc_phase, abort_flag, p, ST_TIMEOUT_EPILOGUE);
      ok = named_bar_and(1, C::EPI_THREADS, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int m = (c.m_blk * 2 + static_cast<int>(rank & 1u)) * C::BM + row;
      const int nbase = c.n_blk * C::BN;
      // The whole row segment comes out of TMEM before any arithmetic and the accumulator is
      // released at once: the next tile's MMAs need all of it, and holding it through the
      // epilogue math stalled them for longer than the math itself takes.
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (is_leader)
            mbar_arrive(bar_tempty);
          else
            tc_commit_pair_mc(bar_tempty, leader_mask);
        }
      };
      // (the NVFP4 output too: holding the only accumulator through its encoding stalled the next
      // tile's MMAs, 8192^3 315 us against 180 us with a 16-bit output)
      uint32_t r[HC];
#pragma unroll
      for (int ch = 0; ch < HC / 32; ++ch)
        tmem_ld_32x32b_x32(t_row + col0 + ch * 32, reinterpret_cast<uint32_t(&)[32]>(r[32 * ch]));
      tmem_ld_wait();
      release();
      epilogue_row<OUT, HC / 16, EXT>(p, c.batch, m, m < p.M, nbase + col0, r, alpha);
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
