// mx_gemm.cuh -- block-scaled GEMMs on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// One warp-specialized, persistent kernel skeleton serves three products, all of the form
// C[m][n] = sum_k A[m][k] B[n][k] with K-contiguous operands:
//   kMxf8 : MXFP8 -- tcgen05.mma kind::mxf8f6f4.block_scale, one E8M0 scale per 32 of K for
//           each operand; the tensor core applies sA_b * sB_b to every 32-block partial sum.
//           "MXFP8 on SM120: software support" (xuesongtap.github.io), sec 0.3.
//   kNvf4 : NVFP4 -- kind::mxf4nvf4.block_scale.scale_vec::4X, one E4M3 scale per 16 of K;
//           the FP32 per-tensor scales multiply the result in the epilogue.
//           "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 7.3 (four-step pipeline:
//           narrow products, per-16 partial sums, times block scales, epilogue times the
//           global scale) and sec 7.4 (scales of both operands).
//   kMxf4 : MXFP4 -- kind::mxf4nvf4.block_scale.scale_vec::2X, E2M1 operands with one E8M0
//           scale per 32 of K (the MX scale layout); "NVFP4: high accuracy with 4 bits"
//           (theluyuan.com), sec 5.5.
//   kDsF8 : DeepSeek FP8 -- kind::f8f6f4 over one 128-wide k-block at a time into one of four
//           TMEM accumulators; epilogue warps promote every k-block into FP32 registers as
//           acc += sA[kb][m] * sB[n/128][kb] * P while the tensor core fills the next buffers.
//           "Why FP8 training is stable" (magicnetworld.com), sec 6.3 (N_C = 128 promotion,
//           overlapped with MMA issue).
//
// Roles (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: A/B tiles (128-byte swizzled rows, one row = 128 B of K) and
//               scale chunks (bulk copies) into a ring of smem stages.
//   warp 1      TMEM allocation + single-thread MMA issue: tcgen05.cp of the stage's scale
//               chunks into TMEM, then 4 tcgen05.mma (32 bytes of K each) per stage.
//   warps 2-9   epilogue, two warps per TMEM lane quarter: tcgen05.ld of the accumulator into
//               registers, release of the accumulator, then scale / convert / vector stores
//               (overlapping the next tile's MMAs).
// Stages are handed over with mbarriers (TMA complete_tx -> MMA; tcgen05.commit -> producer;
// tcgen05.commit -> epilogue; epilogue arrivals -> MMA).  Every wait is bounded.
#pragma once

#include "mx_device.cuh"

namespace mxgb {

enum GemmKind : int { kMxf8 = 0, kNvf4 = 1, kDsF8 = 2, kMxf4 = 3 };

// Bytes of scale chunks a stage needs per 128 rows: MX 1 chunk (128 of K), NVFP4 4 chunks (64 of
// K each), MXFP4 2 chunks (256 of K); DeepSeek scales do not go through shared memory.
constexpr int stage_sf_bytes(int kind) { return kind == kMxf8 ? 512 : (kind == kNvf4 ? 2048 : (kind == kMxf4 ? 1024 : 0)); }
constexpr bool fp4_kind(int kind) { return kind == kNvf4 || kind == kMxf4; }

constexpr int kSmemLimit = 232448;  // 227 KB opt-in dynamic shared memory per CTA

template <int KIND, int BN>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int KBYTES = 128;  // bytes of K per stage: one 128-byte swizzle row
  static constexpr int K_ELEMS = fp4_kind(KIND) ? 256 : 128;
  static constexpr int A_BYTES = BM * KBYTES;
  static constexpr int B_BYTES = BN * KBYTES;
  static constexpr int RC = BN / 128;  // 128-row scale chunks of B per tile
  static constexpr int SFA_BYTES = stage_sf_bytes(KIND);
  static constexpr int SFB_BYTES = SFA_BYTES * RC;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int STAGES_RAW = (kSmemLimit - 1024 - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static constexpr int NUM_MMA = KBYTES / 32;  // tcgen05.mma per stage (32 bytes of K each)
  // TMEM accumulators: one 128 x BN buffer for the block-scaled kinds (the epilogue drains it
  // into registers and releases it at once); four 128-column k-block buffers for DeepSeek.
  static constexpr int NBUF = (KIND == kDsF8) ? 4 : 1;
  static constexpr int ACC_COLS = NBUF * BN;
  // Scale factors get their own TMEM columns per pipeline stage, so the tcgen05.cp of stage s+1
  // carries no write-after-read dependency on the MMAs still reading stage s's scales.
  static constexpr int SFA_COLS = SFA_BYTES / 128;  // one 512-byte chunk fills 4 columns
  static constexpr int SFB_COLS = SFA_COLS * RC;
  static constexpr int SF_STAGE_COLS = SFA_COLS + SFB_COLS;
  static constexpr int SFA_COL = ACC_COLS;             // + stage * SF_STAGE_COLS
  static constexpr int SFB_COL = ACC_COLS + SFA_COLS;  // + stage * SF_STAGE_COLS
  static constexpr int USED_COLS = ACC_COLS + STAGES * SF_STAGE_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 32 ? 32 : USED_COLS <= 64 ? 64 : USED_COLS <= 128 ? 128
                                   : USED_COLS <= 256 ? 256 : 512;
  static constexpr int NUM_EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half of BN
  static constexpr bool HAS_SF = (KIND != kDsF8);
  static constexpr int SF_WARP = 2 + NUM_EPI_WARPS;  // issues the scale copies (block-scaled kinds)
  static constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS + (HAS_SF ? 32 : 0);
  static constexpr int EPI_THREADS = 32 * NUM_EPI_WARPS;
  static_assert(STAGES >= 2, "not enough shared memory for two stages");
  static_assert(USED_COLS <= 512, "TMEM overflow");
  static_assert(KIND != kDsF8 || BN == 128, "the promotion epilogue holds 64 columns per thread");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "bad BN");
};

struct GemmArgs {
  const uint8_t* sfa;  // MX / NV scale chunks of A
  const uint8_t* sfb;
  const float* dsa;  // DeepSeek: float[K/128][M]
  const float* dsb;  // DeepSeek: float[N/128][K/128]
  const float* ga;   // NVFP4 global scales
  const float* gb;
  int ga_stride;     // grouped NVFP4: 0 = one global scale of A, 1 = one per group (ga[g])
  void* out;
  int64_t ldc;
  int M, N, K;  // K in elements (grouped: M = rows of all groups)
  uint32_t idesc;
  const int64_t* group_off;  // grouped GEMM: device int64[groups + 1] row offsets of the groups
  int groups;
  uint8_t* q_out;  // MX output, row-wise: codes [M][ldc bytes] and E8M0 scales in the MX GEMM
  uint8_t* s_out;  // layout (either may be skipped by passing null codes)
  uint8_t* q_col;  // MX output, column-wise: codes [N][ldq_col bytes] (the transpose of the
  uint8_t* s_col;  // result, blocks of 32 rows) and E8M0 scales in the MX GEMM layout of [N][M]
  int64_t ldq_col;
};

constexpr int kMaxGroups = 1024;

// Tile order: bands of 16 m-blocks; inside a band, m runs fastest, so the CTAs of one wave
// share a few B tiles and a band of A tiles in L2.
__device__ __forceinline__ void tile_coords(int tile, int num_mb, int num_nb, int& mb, int& nb) {
  constexpr int G = 16;
  const int band_tiles = G * num_nb;
  const int band = tile / band_tiles;
  const int in = tile - band * band_tiles;
  const int mb0 = band * G;
  const int gm = min(G, num_mb - mb0);
  nb = in / gm;
  mb = mb0 + (in - nb * gm);
}

template <bool OUT_BF16>
__device__ __forceinline__ void store_row32(void* out, int64_t ldc, int64_t row, int64_t col, const float* v) {
  if (OUT_BF16) {
    uint32_t p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      p[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row * ldc + col);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row * ldc + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

template <int KIND, int BN, bool OUT_BF16>
__global__ void __launch_bounds__(GemmCfg<KIND, BN>::THREADS, 1)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args) {
  using Cfg = GemmCfg<KIND, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + Cfg::STAGES * Cfg::A_BYTES;
  uint8_t* sSFA = sB + Cfg::STAGES * Cfg::B_BYTES;
  uint8_t* sSFB = sSFA + Cfg::STAGES * Cfg::SFA_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSFB + Cfg::STAGES * Cfg::SFB_BYTES);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + Cfg::STAGES;
  uint64_t* tfull_bar = bars + 2 * Cfg::STAGES;       // [NBUF]
  uint64_t* tempty_bar = bars + 2 * Cfg::STAGES + 4;  // [NBUF]
  uint64_t* drain_bar = bars + 2 * Cfg::STAGES + 8;
  uint64_t* sfdrain_bar = bars + 2 * Cfg::STAGES + 9;
  uint64_t* sfready_bar = bars + 2 * Cfg::STAGES + 10;  // [STAGES]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * Cfg::STAGES + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_mb = args.M / Cfg::BM;
  const int num_nb = args.N / BN;
  const int num_tiles = num_mb * num_nb;
  const int num_kt = args.K / Cfg::K_ELEMS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < Cfg::NBUF; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], Cfg::EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    mbar_init(sfdrain_bar, 1);
    for (int st = 0; st < Cfg::STAGES; ++st) mbar_init(&sfready_bar[st], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      const int64_t kchunks_mx = args.K / 128;  // MX scale chunks per 128 rows
      const int64_t kchunks_nv = args.K / 64;   // NV scale chunks per 128 rows
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_mb, num_nb, mb, nb);
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
          tma_load_2d(sA + stage * Cfg::A_BYTES, &tmA, &full_bar[stage], kt * Cfg::KBYTES, mb * Cfg::BM);
          tma_load_2d(sB + stage * Cfg::B_BYTES, &tmB, &full_bar[stage], kt * Cfg::KBYTES, nb * BN);
          if (KIND == kMxf8) {
            bulk_load(sSFA + stage * Cfg::SFA_BYTES, args.sfa + (mb * kchunks_mx + kt) * 512, 512,
                      &full_bar[stage]);
#pragma unroll
            for (int rc = 0; rc < Cfg::RC; ++rc)
              bulk_load(sSFB + stage * Cfg::SFB_BYTES + rc * 512,
                        args.sfb + ((static_cast<int64_t>(nb) * Cfg::RC + rc) * kchunks_mx + kt) * 512, 512,
                        &full_bar[stage]);
          } else if (KIND == kMxf4) {  // MX chunks 2kt, 2kt + 1: 1 KB per 128 rows
            bulk_load(sSFA + stage * Cfg::SFA_BYTES, args.sfa + (mb * kchunks_mx + 2ll * kt) * 512, 1024,
                      &full_bar[stage]);
#pragma unroll
            for (int rc = 0; rc < Cfg::RC; ++rc)
              bulk_load(sSFB + stage * Cfg::SFB_BYTES + rc * 1024,
                        args.sfb + ((static_cast<int64_t>(nb) * Cfg::RC + rc) * kchunks_mx + 2ll * kt) * 512, 1024,
                        &full_bar[stage]);
          } else if (KIND == kNvf4) {
            bulk_load(sSFA + stage * Cfg::SFA_BYTES, args.sfa + (mb * kchunks_nv + 4ll * kt) * 512, 2048,
                      &full_bar[stage]);
#pragma unroll
            for (int rc = 0; rc < Cfg::RC; ++rc)
              bulk_load(sSFB + stage * Cfg::SFB_BYTES + rc * 2048,
                        args.sfb + ((static_cast<int64_t>(nb) * Cfg::RC + rc) * kchunks_nv + 4ll * kt) * 512, 2048,
                        &full_bar[stage]);
          }
          ++issued;
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: every copy this thread issued must have landed before the CTA exits
      for (int s = 0; s < Cfg::STAGES; ++s) {
        if (issued > s) {
          const long last = s + ((issued - 1 - s) / Cfg::STAGES) * Cfg::STAGES;
          mbar_wait(&full_bar[s], static_cast<uint32_t>((last / Cfg::STAGES) & 1), abort_flag, kSiteDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The issue path of this single thread bounds the CTA's throughput, so per k-step it does only:
    // the barrier waits, the MMAs with descriptor words advanced by constants, and the commits.
    // The scale copies come from another warp: they overlap the MMAs only when a different thread
    // issues them.
    if (lane == 0) {
      constexpr uint32_t kOpHi = smem_desc_hi(1024, kSwizzle128B);
      constexpr uint32_t kLbo = smem_desc_lo_lbo(16);
      const uint32_t a_lo0 = (smem_u32(sA) >> 4) | kLbo, b_lo0 = (smem_u32(sB) >> 4) | kLbo;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_it = 0;  // accumulator hand-overs so far
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (KIND != kDsF8) {
          if (!mbar_wait(&tempty_bar[0], (acc_it & 1) ^ 1, abort_flag, kSiteMmaTmemEmpty)) break;
          tc_fence_after();
        }
        for (int kt = 0; kt < num_kt; ++kt) {
          uint32_t d_tmem = tmem_base;
          if (KIND == kDsF8) {
            const uint32_t b = acc_it % Cfg::NBUF;
            if (!mbar_wait(&tempty_bar[b], ((acc_it / Cfg::NBUF) & 1) ^ 1, abort_flag, kSiteMmaTmemEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + b * BN;
          }
          // block-scaled kinds wait for the scale-copy warp's stage barrier (it follows the TMA
          // barrier), the promotion kind for the TMA barrier itself
          if (!mbar_wait(Cfg::HAS_SF ? &sfready_bar[stage] : &full_bar[stage], phase, abort_flag, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_lo = a_lo0 + stage * (Cfg::A_BYTES >> 4);
          const uint32_t b_lo = b_lo0 + stage * (Cfg::B_BYTES >> 4);
          const uint32_t sfa_t = tmem_base + Cfg::SFA_COL + stage * Cfg::SF_STAGE_COLS;
          const uint32_t sfb_t = tmem_base + Cfg::SFB_COL + stage * Cfg::SF_STAGE_COLS;
#pragma unroll
          for (int j = 0; j < Cfg::NUM_MMA; ++j) {
            const uint64_t adesc = desc_from_words(a_lo + j * 2, kOpHi);  // + 32 bytes of K per MMA
            const uint64_t bdesc = desc_from_words(b_lo + j * 2, kOpHi);
            if (KIND == kMxf8) {
              umma_mxf8f6f4(d_tmem, adesc, bdesc, idesc_with_sf_ids(args.idesc, j, j), sfa_t, sfb_t,
                            (kt > 0 || j > 0) ? 1u : 0u);
            } else if (KIND == kMxf4) {  // MMA j: scale chunk j / 2, bytes 2 (j % 2) .. + 1 of each row
              umma_mxf4(d_tmem, adesc, bdesc, idesc_with_sf_ids(args.idesc, 2 * (j & 1), 2 * (j & 1)),
                        sfa_t + 4 * (j >> 1), sfb_t + (j >> 1) * 4 * Cfg::RC, (kt > 0 || j > 0) ? 1u : 0u);
            } else if (KIND == kNvf4) {
              umma_mxf4nvf4(d_tmem, adesc, bdesc, args.idesc, sfa_t + 4 * j, sfb_t + j * 4 * Cfg::RC,
                            (kt > 0 || j > 0) ? 1u : 0u);
            } else {
              umma_f8f6f4(d_tmem, adesc, bdesc, args.idesc, j > 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty_bar[stage]);  // frees the smem stage once these MMAs are done
          if (KIND == kDsF8) {
            umma_commit(&tfull_bar[acc_it % Cfg::NBUF]);  // one k-block ready for promotion
            ++acc_it;
          }
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (KIND != kDsF8 && ok) {
          umma_commit(&tfull_bar[0]);
          ++acc_it;
        }
      }
      // drain: all MMAs issued by this thread complete before TMEM is released
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, abort_flag, kSiteDrain);
    }
  } else if (Cfg::HAS_SF && warp == Cfg::SF_WARP) {
    // ------------------------------------------------------------------ scale copies
    if (lane == 0) {
      constexpr uint32_t kSfHi = smem_desc_hi(128, kSwizzleNone);
      const uint32_t sfa_lo0 = smem_u32(sSFA) >> 4, sfb_lo0 = smem_u32(sSFB) >> 4;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_lo = sfa_lo0 + stage * (Cfg::SFA_BYTES >> 4);
          const uint32_t sfb_lo = sfb_lo0 + stage * (Cfg::SFB_BYTES >> 4);
          const uint32_t sfa_t = tmem_base + Cfg::SFA_COL + stage * Cfg::SF_STAGE_COLS;
          const uint32_t sfb_t = tmem_base + Cfg::SFB_COL + stage * Cfg::SF_STAGE_COLS;
          if (KIND == kMxf8) {
            tmem_cp_32x128b_warpx4(sfa_t, desc_from_words(sfa_lo, kSfHi));
#pragma unroll
            for (int rc = 0; rc < Cfg::RC; ++rc)
              tmem_cp_32x128b_warpx4(sfb_t + 4 * rc, desc_from_words(sfb_lo + rc * (512 >> 4), kSfHi));
          } else {
            // chunk c of A's scales -> columns 4c; chunk c of B's row block rc -> 4 (c RC + rc)
            constexpr int NCH = Cfg::SFA_BYTES / 512;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
              tmem_cp_32x128b_warpx4(sfa_t + 4 * c, desc_from_words(sfa_lo + c * (512 >> 4), kSfHi));
#pragma unroll
              for (int rc = 0; rc < Cfg::RC; ++rc)
                tmem_cp_32x128b_warpx4(sfb_t + c * 4 * Cfg::RC + 4 * rc,
                                       desc_from_words(sfb_lo + ((rc * Cfg::SFA_BYTES + c * 512) >> 4), kSfHi));
            }
          }
          umma_commit(&sfready_bar[stage]);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: every copy this thread issued completes before TMEM is released
      umma_commit(sfdrain_bar);
      mbar_wait(sfdrain_bar, 0, abort_flag, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the BN columns this warp owns
    const int row_in_tile = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint32_t acc_it = 0;
    if (KIND != kDsF8) {
      constexpr int HALF = BN / 2;
      constexpr int NCH = HALF / 32;
      float gscale = 1.0f;
      if (KIND == kNvf4) gscale = __fmul_rn(*args.ga, *args.gb);
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_mb, num_nb, mb, nb);
        bool ok = mbar_wait(&tfull_bar[0], acc_it & 1, abort_flag, kSiteEpiTmemFull);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        tc_fence_after();
        // drain this warp's 32 rows x HALF columns into registers, then hand the accumulator
        // back so the next tile's MMAs overlap the conversion and the stores below
        uint32_t r[NCH][32];
#pragma unroll
        for (int c = 0; c < NCH; ++c) tmem_ld_32x32b_x32(tmem_base + lane_addr + half * HALF + c * 32, r[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < NCH; ++c) tmem_regs_ready(r[c]);
        tc_fence_before();
        mbar_arrive(&tempty_bar[0]);
        ++acc_it;
        const int64_t row = static_cast<int64_t>(mb) * Cfg::BM + row_in_tile;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = (KIND == kNvf4) ? __fmul_rn(__uint_as_float(r[c][i]), gscale) : __uint_as_float(r[c][i]);
          store_row32<OUT_BF16>(args.out, args.ldc, row, static_cast<int64_t>(nb) * BN + half * HALF + c * 32, v);
        }
      }
    } else {
      // DeepSeek promotion: this warp owns rows q*32.. and columns [half*64, half*64+64).  K-blocks
      // are promoted two at a time: both TMEM buffers are loaded before one wait, so one round trip
      // (barrier wait, TMEM load, release) serves two k-blocks; each k-block still gets its own
      // scale, in order.  The scales are loaded one pair ahead so their latency hides too.
      const int64_t kbs = args.K / 128;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_mb, num_nb, mb, nb);
        const int64_t row = static_cast<int64_t>(mb) * Cfg::BM + row_in_tile;
        const float* sa_row = args.dsa + row;
        const float* sb_blk = args.dsb + static_cast<int64_t>(nb) * kbs;
        float nsa0 = __ldg(sa_row), nsb0 = __ldg(sb_blk);
        float nsa1 = 0.0f, nsb1 = 0.0f;
        if (num_kt > 1) {
          nsa1 = __ldg(sa_row + args.M);
          nsb1 = __ldg(sb_blk + 1);
        }
        uint64_t acc[32];  // 64 FP32 accumulators as pairs, updated with paired FMAs
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0ull;
        for (int kt = 0; kt < num_kt; kt += 2) {
          const bool two = kt + 1 < num_kt;
          const float s0 = __fmul_rn(nsa0, nsb0), s1 = __fmul_rn(nsa1, nsb1);
          if (kt + 2 < num_kt) {
            nsa0 = __ldg(sa_row + static_cast<int64_t>(kt + 2) * args.M);
            nsb0 = __ldg(sb_blk + kt + 2);
          }
          if (kt + 3 < num_kt) {
            nsa1 = __ldg(sa_row + static_cast<int64_t>(kt + 3) * args.M);
            nsb1 = __ldg(sb_blk + kt + 3);
          }
          const uint32_t b0 = acc_it % Cfg::NBUF, b1 = (acc_it + 1) % Cfg::NBUF;
          ok = mbar_wait(&tfull_bar[b0], (acc_it / Cfg::NBUF) & 1, abort_flag, kSiteEpiTmemFull);
          if (two) ok = ok && mbar_wait(&tfull_bar[b1], ((acc_it + 1) / Cfg::NBUF) & 1, abort_flag, kSiteEpiTmemFull);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t r0[32], r1[32];
          const uint32_t t0 = tmem_base + lane_addr + b0 * BN + half * 64;
          const uint32_t t1 = tmem_base + lane_addr + b1 * BN + half * 64;
          tmem_ld_32x32b_x32(t0, r0);
          tmem_ld_32x32b_x32(t0 + 32, r1);
          tmem_ld_wait();
          tmem_regs_ready(r0);
          tmem_regs_ready(r1);
          tc_fence_before();
          mbar_arrive(&tempty_bar[b0]);
          // the second k-block's TMEM loads overlap the first one's FMAs
          const uint64_t s0x2 = pack_f32x2(s0, s0), s1x2 = pack_f32x2(s1, s1);
#pragma unroll
          for (int i = 0; i < 16; ++i) fma2_scalar(acc[i], s0x2, r0[2 * i], r0[2 * i + 1]);
          if (two) tmem_ld_32x32b_x32(t1, r0);
#pragma unroll
          for (int i = 0; i < 16; ++i) fma2_scalar(acc[16 + i], s0x2, r1[2 * i], r1[2 * i + 1]);
          if (two) {
            tmem_ld_32x32b_x32(t1 + 32, r1);
            tmem_ld_wait();
            tmem_regs_ready(r0);
            tmem_regs_ready(r1);
            tc_fence_before();
            mbar_arrive(&tempty_bar[b1]);
#pragma unroll
            for (int i = 0; i < 16; ++i) fma2_scalar(acc[i], s1x2, r0[2 * i], r0[2 * i + 1]);
#pragma unroll
            for (int i = 0; i < 16; ++i) fma2_scalar(acc[16 + i], s1x2, r1[2 * i], r1[2 * i + 1]);
          }
          acc_it += two ? 2 : 1;
        }
        if (!ok) break;
        float accf[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) unpack_f32x2(acc[i], accf[2 * i], accf[2 * i + 1]);
        store_row32<OUT_BF16>(args.out, args.ldc, row, static_cast<int64_t>(nb) * BN + half * 64, accf);
        store_row32<OUT_BF16>(args.out, args.ldc, row, static_cast<int64_t>(nb) * BN + half * 64 + 32, accf + 32);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

}  // namespace mxgb
