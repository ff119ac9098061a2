// mx_gemm2.cuh -- block-scaled GEMMs on CTA pairs (tcgen05 cta_group::2) for sm_103a.
//
// Same products as the single-CTA kernel (kMxf8: MXFP8 with E8M0 scales per 32 of K; kMxf4:
// MXFP4, E2M1 with E8M0 scales per 32; kNvf4: NVFP4 with E4M3 scales per 16 and FP32 global
// scales in the epilogue), but one 256 x 256 output
// tile is computed by a cluster of two CTAs on two SMs with M = 256 tcgen05.mma instructions:
//   * each CTA loads its own 128 rows of A and its own 128 rows (half) of B per stage; the pair's
//     MMA reads both halves of B, so every SM receives 2/3 of the operand bytes the single-CTA
//     128 x 256 tile needs for the same number of MACs;
//   * each CTA holds the scales of its 128 rows of A and the scales of all 256 rows of B; one
//     pair-wide tcgen05.cp copies every CTA's scales from its own shared memory into its own TMEM,
//     so the scale copies per MAC halve as well;
//   * the leader CTA (rank 0) issues the MMAs and scale copies for the pair; both CTAs' TMA loads
//     complete on the leader's stage barrier; the leader's commits arrive on the stage and
//     accumulator barriers of both CTAs; both CTAs' epilogues drain their own TMEM accumulator
//     (their 128 rows x 256 columns) and arrive on the leader's accumulator-free barrier.
// Sources: "MXFP8 on SM120: software support" (xuesongtap.github.io), sec 0.3 (block-scaled
// dot product); "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 7.3-7.4.
#pragma once

#include "mx_device.cuh"
#include "mx_gemm.cuh"

namespace mxgb {

// Write one warp's 32 x 32 output chunk (row = lane, 32 consecutive columns in v) through its
// swizzled staging buffer and one TMA tensor store at (x, y) -- fewer, larger writes than
// per-thread vector stores, which slowed the MMA issue.  The buffer is reused only after the
// previous store has read it.
template <bool OUT_BF16>
__device__ __forceinline__ void store_chunk_32x32(const CUtensorMap* tmOut, uint8_t* buf, const float (&v)[32],
                                                  int lane, int32_t x, int32_t y) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  if (OUT_BF16) {
    // 32 rows x 64 B, 64-byte swizzle: 16-byte piece k of row r sits at piece k ^ ((r >> 1) & 3)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * k + 2 * e], v[8 * k + 2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(buf + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    // 32 rows x 128 B, 128-byte swizzle: piece k of row r sits at piece k ^ (r & 7)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<float4*>(buf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
          make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmOut, buf, x, y);
    bulk_commit_group();
  }
}

// Grouped products: per-group first tile numbers (tiles numbered group by group, each group's
// rows in BM-row tiles times num_nb column tiles).  Offsets must start at 0, end at M, be
// multiples of 128 and never decrease; otherwise every entry is 0 (no tile runs) and the error
// word reports it.  One thread fills the table; the caller synchronizes before others read it.
__device__ __forceinline__ void build_group_table(int* grp_start, const GemmArgs& args, int bm, int num_nb) {
  const int64_t* off = args.group_off;
  bool good = __ldg(off) == 0 && __ldg(off + args.groups) == args.M;
  int t = 0;
  for (int g = 0; g < args.groups; ++g) {
    grp_start[g] = t;
    const int64_t a = __ldg(off + g), b = __ldg(off + g + 1);
    good = good && a >= 0 && b >= a && (a & 127) == 0 && (b & 127) == 0 && b <= args.M;
    if (good) t += static_cast<int>((b - a + bm - 1) / bm) * num_nb;
  }
  if (!good) {
    t = 0;
    if (blockIdx.x == 0) atomicOr(&g_mx_error_word, kSiteBadGroups);
  }
  grp_start[args.groups] = t;
}

// Grouped tile -> group, first A row of the tile, first row of B (the experts' blocks stacked),
// rows of the group from a_row0 on (at most bm), column tile.
__device__ __forceinline__ void decode_group_tile(const int* grp_start, const GemmArgs& args, int bm, int bn,
                                                  int num_nb, int tile, int& grp, int64_t& a_row0, int64_t& b_row0,
                                                  int& rows_valid, int& nb) {
  int lo = 0, hi = args.groups - 1;  // the last group whose first tile is <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (grp_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  const int64_t off = __ldg(args.group_off + lo), rows_g = __ldg(args.group_off + lo + 1) - off;
  int mb;
  tile_coords(tile - grp_start[lo], static_cast<int>((rows_g + bm - 1) / bm), num_nb, mb, nb);
  a_row0 = off + static_cast<int64_t>(mb) * bm;
  b_row0 = static_cast<int64_t>(lo) * args.N + static_cast<int64_t>(nb) * bn;
  const int64_t left = rows_g - static_cast<int64_t>(mb) * bm;
  rows_valid = left < bm ? static_cast<int>(left) : bm;
  grp = lo;
}

// byte offset of row i's 4 scale bytes inside a 512-byte MX scale chunk
__device__ __forceinline__ int chunk_offset_mx(int i) { return (i & 31) * 16 + (i >> 5) * 4; }

// NARROW_OUT: bf16 (or MX codes) out, whose 32 x 32 staging chunk is 2 KB instead of FP32's 4 KB;
// the freed shared memory holds one more pipeline stage for MXFP8 (6 instead of 5: +3-5%).
template <int KIND, bool NARROW_OUT = false, bool GROUPED_ = false>
struct Gemm2Cfg {
  static constexpr int BM = 256;       // rows per pair tile (128 per CTA)
  static constexpr int BN = 256;       // columns per pair tile
  static constexpr int ROWS = 128;     // A rows and B rows each CTA loads
  static constexpr int KBYTES = 128;   // bytes of K per stage
  static constexpr int K_ELEMS = fp4_kind(KIND) ? 256 : 128;
  static constexpr int A_BYTES = ROWS * KBYTES;
  static constexpr int B_BYTES = ROWS * KBYTES;
  static constexpr int SF_CHUNK = stage_sf_bytes(KIND);  // scale bytes per 128 rows per stage
  static constexpr int SFA_BYTES = SF_CHUNK;       // own 128 rows of A
  static constexpr int SFB_BYTES = 2 * SF_CHUNK;   // all 256 rows of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int BAR_BYTES = 1024;
  // output staging for the TMA stores: one 32 x 32 chunk per epilogue warp, 1 KB aligned for the
  // 128-byte swizzle
  static constexpr int CHUNK_BYTES = NARROW_OUT ? 2048 : 4096;
  static constexpr int STAGING = 8 * CHUNK_BYTES + 1024;
  // static shared memory of the kernel (the grouped kernels' table of group start tiles) comes
  // out of the same per-CTA limit
  static constexpr int STATIC_SMEM = GROUPED_ ? (kMaxGroups + 1) * 4 + 64 : 64;
  static constexpr int STAGES_RAW = (kSmemLimit - 1024 - BAR_BYTES - STAGING - STATIC_SMEM) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING + BAR_BYTES;
  static constexpr int NUM_MMA = KBYTES / 32;
  static constexpr int ACC_COLS = BN;
  static constexpr int SFA_COLS = SF_CHUNK / 128;  // a 512-byte chunk fills 4 TMEM columns
  static constexpr int SFB_COLS = 2 * SFA_COLS;
  static constexpr int SF_STAGE_COLS = SFA_COLS + SFB_COLS;  // each stage has its own scale columns
  static constexpr int SFA_COL = ACC_COLS;                     // + stage * SF_STAGE_COLS
  static constexpr int SFB_COL = ACC_COLS + SFA_COLS;          // + stage * SF_STAGE_COLS
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_EPI_WARPS = 8;
  // warps SF_WARP .. SF_WARP + SF_ISSUERS - 1 issue the scale copies (leader CTA): one thread
  // cannot issue the twelve NVFP4 copies of a stage as fast as the MMAs consume them
  static constexpr int SF_WARP = 2 + NUM_EPI_WARPS;
  static constexpr int SF_ISSUERS = 2;
  static constexpr int THREADS = 64 + 32 * SF_ISSUERS + 32 * NUM_EPI_WARPS;
  static constexpr int EPI_THREADS = 32 * NUM_EPI_WARPS;
  static_assert(STAGES >= 2, "not enough shared memory");
  static_assert(ACC_COLS + STAGES * SF_STAGE_COLS <= TMEM_COLS, "TMEM overflow");
};

// Scale tensors are read through 2-D byte tensor maps with 128-byte rows (a 512-byte scale chunk
// is 4 such rows), so that the peer CTA's scale loads can complete on the leader's barrier too.
// GROUPED (MoE expert GEMMs in one launch; "MXFP8 on SM120: software support"
// (xuesongtap.github.io), sec 1.2: grouped GEMM is its own entry point): group g multiplies rows
// off[g] .. off[g+1] of A by the g-th [N][K] block of B into the same rows of C (NVFP4: times
// s_gA * s_gB[g], each expert's weights having their own global scale); tiles are
// numbered group by group (the per-group tile counts' prefix sums sit in shared memory) and a
// CTA whose 128 rows lie past its group's last row computes but stores nothing.
// MXOUT >= 0: the epilogue quantizes its FP32 results itself with the MX rule and writes codes
// and E8M0 scales instead of bf16 / FP32 values -- the producer-side fusion of the next layer's
// quantization ("Why FP8 training is stable" (magicnetworld.com), sec 9: the activations feeding
// the next FP8 product are quantized before they leave).  MXOUT = format + 2 * copies: format 0
// E4M3, 1 E5M2; copies 1 row-wise (1x32 blocks, the next product's A operand), 2 column-wise
// (32x1 blocks, stored transposed: the operand of a product reducing over M), 3 both.  Each copy
// is compiled in only where it is written.
constexpr int mxout_code(int fmt, int copies) { return fmt + 2 * copies; }
template <int KIND, bool OUT_BF16, bool GROUPED = false, int MXOUT = -1>
__global__ void __launch_bounds__(Gemm2Cfg<KIND, OUT_BF16 || (MXOUT >= 0), GROUPED>::THREADS, 1)
    bs_gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                    const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
  using Cfg = Gemm2Cfg<KIND, OUT_BF16 || (MXOUT >= 0), GROUPED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + Cfg::STAGES * Cfg::A_BYTES;
  uint8_t* sSFA = sB + Cfg::STAGES * Cfg::B_BYTES;
  uint8_t* sSFB = sSFA + Cfg::STAGES * Cfg::SFA_BYTES;
  uint8_t* sOut = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sSFB + Cfg::STAGES * Cfg::SFB_BYTES) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSFB + Cfg::STAGES * Cfg::SFB_BYTES + Cfg::STAGING);
  uint64_t* full_bar = bars;                       // [STAGES], used in the leader
  uint64_t* empty_bar = bars + Cfg::STAGES;        // [STAGES], both CTAs
  uint64_t* tfull_bar = bars + 2 * Cfg::STAGES;    // both CTAs
  uint64_t* tempty_bar = tfull_bar + 1;            // used in the leader
  uint64_t* drain_bar = tfull_bar + 2;
  uint64_t* sfready_bar = tfull_bar + 3;           // [STAGES], used in the leader
  uint64_t* sfdrain_bar = tfull_bar + 3 + Cfg::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull_bar + 4 + Cfg::STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int num_mb = args.M / Cfg::BM;
  const int num_nb = args.N / Cfg::BN;
  const int num_kt = args.K / Cfg::K_ELEMS;
  __shared__ int grp_start[GROUPED ? kMaxGroups + 1 : 1];  // first tile of each group
  if (GROUPED && threadIdx.x == 0) build_group_table(grp_start, args, Cfg::BM, num_nb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * Cfg::EPI_THREADS);
    mbar_init(drain_bar, 1);
    for (int st = 0; st < Cfg::STAGES; ++st) mbar_init(&sfready_bar[st], Cfg::SF_ISSUERS);
    mbar_init(sfdrain_bar, Cfg::SF_ISSUERS);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
    prefetch_tmap(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = GROUPED ? grp_start[args.groups] : num_mb * num_nb;
  // tile -> (first A row, first B row, rows of A that belong to it, output column block)
  auto decode = [&](int tile, int64_t& a_row0, int64_t& b_row0, int& rows_valid, int& nb, int& grp) {
    grp = 0;
    if (GROUPED) {
      decode_group_tile(grp_start, args, Cfg::BM, Cfg::BN, num_nb, tile, grp, a_row0, b_row0, rows_valid, nb);
    } else {
      int mb;
      tile_coords(tile, num_mb, num_nb, mb, nb);
      a_row0 = static_cast<int64_t>(mb) * Cfg::BM;
      b_row0 = static_cast<int64_t>(nb) * Cfg::BN;
      rows_valid = Cfg::BM;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      const int64_t kc = (KIND == kNvf4) ? args.K / 64 : args.K / 128;  // 512-byte chunks per 128 rows
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
        int64_t a_row0, b_row0;
        int rows_valid, nb, grp;
        decode(tile, a_row0, b_row0, rows_valid, nb, grp);
        const int a_row = static_cast<int>(a_row0) + static_cast<int>(rank) * Cfg::ROWS;
        const int b_row = static_cast<int>(b_row0) + static_cast<int>(rank) * Cfg::ROWS;
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = map_to_rank(smem_u32(&full_bar[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * Cfg::STAGE_BYTES);
          tma_load_2d_pair(sA + stage * Cfg::A_BYTES, &tmA, full_leader, kt * Cfg::KBYTES, a_row);
          tma_load_2d_pair(sB + stage * Cfg::B_BYTES, &tmB, full_leader, kt * Cfg::KBYTES, b_row);
          // 512-byte scale chunk (rb, c) starts at 128-byte row (rb * kc + c) * 4; a stage needs
          // chunk c = kt (MXFP8), chunks 2kt, 2kt+1 (MXFP4) or 4kt .. 4kt+3 (NVFP4), contiguous,
          // so one box
          const int64_t cfirst = static_cast<int64_t>(Cfg::SF_CHUNK / 512) * kt;
          tma_load_2d_pair(sSFA + stage * Cfg::SFA_BYTES, &tmSFA, full_leader, 0,
                           static_cast<int32_t>(((a_row / 128) * kc + cfirst) * 4));
#pragma unroll
          for (int rc = 0; rc < 2; ++rc)
            tma_load_2d_pair(sSFB + stage * Cfg::SFB_BYTES + rc * Cfg::SF_CHUNK, &tmSFB, full_leader, 0,
                             static_cast<int32_t>(((b_row0 / 128 + rc) * kc + cfirst) * 4));
          ++issued;
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: the leader's stage barriers count both CTAs' bytes, so the leader waits for every
      // copy either CTA issued; the final cluster barrier keeps the peer alive until then
      if (leader) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
          if (issued > s) {
            const long last = s + ((issued - 1 - s) / Cfg::STAGES) * Cfg::STAGES;
            mbar_wait(&full_bar[s], static_cast<uint32_t>((last / Cfg::STAGES) & 1), abort_flag, kSiteDrain);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      // The issue path of this single thread bounds the pair's throughput, so per k-step it does
      // only: one barrier wait, the MMAs with descriptor words advanced by constants, one commit.
      // The scale copies come from another warp (they overlap the MMAs only when a different
      // thread issues them); its per-stage barrier also guarantees the stage's operands landed.
      constexpr uint32_t kOpHi = smem_desc_hi(1024, kSwizzle128B);
      constexpr uint32_t kLbo = smem_desc_lo_lbo(16);
      const uint32_t a_lo0 = (smem_u32(sA) >> 4) | kLbo, b_lo0 = (smem_u32(sB) >> 4) | kLbo;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_it = 0;
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
        if (!mbar_wait(tempty_bar, (acc_it & 1) ^ 1, abort_flag, kSiteMmaTmemEmpty)) break;
        tc_fence_after();
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&sfready_bar[stage], phase, abort_flag, kSiteMmaFull)) {
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
            const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
            if (KIND == kMxf8)
              umma_mxf8f6f4_pair(tmem_base, adesc, bdesc, idesc_with_sf_ids(args.idesc, j, j), sfa_t, sfb_t, acc);
            else if (KIND == kMxf4)  // MMA j: scale chunk j / 2, bytes 2 (j % 2) .. + 1 of each row
              umma_mxf4_pair(tmem_base, adesc, bdesc, idesc_with_sf_ids(args.idesc, 2 * (j & 1), 2 * (j & 1)),
                             sfa_t + 4 * (j >> 1), sfb_t + 8 * (j >> 1), acc);
            else
              umma_mxf4nvf4_pair(tmem_base, adesc, bdesc, args.idesc, sfa_t + 4 * j, sfb_t + 8 * j, acc);
          }
          umma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) {
          umma_commit_pair(tfull_bar, 0x3);
          ++acc_it;
        }
      }
      umma_commit_pair(drain_bar, 0x1);
      mbar_wait(drain_bar, 0, abort_flag, kSiteDrain);
    }
  } else if (warp >= Cfg::SF_WARP) {
    // ------------------------------------------------------------------ scale copies (leader only)
    // Per stage and MMA j there are three 512-byte chunk copies: A's scales, then B's scales for
    // rows 0-127 and 128-255.  Copy c = 3j + w goes to issuer c % SF_ISSUERS.
    const int part = warp - Cfg::SF_WARP;
    if (leader && lane == 0) {
      constexpr uint32_t kSfHi = smem_desc_hi(128, kSwizzleNone);
      const uint32_t sfa_lo0 = smem_u32(sSFA) >> 4, sfb_lo0 = smem_u32(sSFB) >> 4;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
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
          // an MXFP8 stage's four MMAs read one chunk of each scale tensor (bytes picked by the
          // scale ids), an MXFP4 stage's read two (one per pair of MMAs), an NVFP4 stage's four
          constexpr int NCOPY = 3 * (Cfg::SF_CHUNK / 512);
#pragma unroll
          for (int c = 0; c < NCOPY; ++c) {
            if (c % Cfg::SF_ISSUERS != part) continue;
            const int j = c / 3, w = c % 3;
            const uint32_t taddr = (w == 0) ? sfa_t + 4 * j : sfb_t + 8 * j + 4 * (w - 1);
            const uint32_t lo = (w == 0) ? sfa_lo + j * (512 >> 4) : sfb_lo + (((w - 1) * Cfg::SF_CHUNK + j * 512) >> 4);
            tmem_cp_32x128b_warpx4_pair(taddr, desc_from_words(lo, kSfHi));
          }
          umma_commit_pair(&sfready_bar[stage], 0x1);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: every copy this thread issued completes before TMEM is released
      umma_commit_pair(sfdrain_bar, 0x1);
      mbar_wait(sfdrain_bar, 0, abort_flag, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tempty_leader = map_to_rank(smem_u32(tempty_bar), 0);
    constexpr int HALF = Cfg::BN / 2;
    constexpr int NCH = HALF / 32;
    float gscale = 1.0f;
    if (KIND == kNvf4 && !GROUPED) gscale = __fmul_rn(*args.ga, *args.gb);
    uint32_t acc_it = 0;
    for (int tile = cluster; tile < num_tiles; tile += nclusters) {
      int64_t a_row0, b_row0;
      int rows_valid, nb, grp;
      decode(tile, a_row0, b_row0, rows_valid, nb, grp);
      // grouped NVFP4: every expert's B carries its own global scale
      if (KIND == kNvf4 && GROUPED) gscale = __fmul_rn(__ldg(args.ga + grp * args.ga_stride), __ldg(args.gb + grp));
      const bool store = static_cast<int>(rank) * Cfg::ROWS < rows_valid;  // this CTA's rows exist
      bool ok = mbar_wait(tfull_bar, acc_it & 1, abort_flag, kSiteEpiTmemFull);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      uint32_t r[NCH][32];
#pragma unroll
      for (int c = 0; c < NCH; ++c) tmem_ld_32x32b_x32(tmem_base + lane_addr + half * HALF + c * 32, r[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < NCH; ++c) tmem_regs_ready(r[c]);
      tc_fence_before();
      mbar_arrive_cluster(tempty_leader);
      ++acc_it;
      // each 32 x 32 chunk goes through this warp's swizzled staging buffer and one TMA store
      // (fewer, larger writes than per-thread vector stores, which slowed the MMA issue)
      uint8_t* buf = sOut + (warp - 2) * Cfg::CHUNK_BYTES;
      const int32_t y0 = static_cast<int32_t>(a_row0 + rank * Cfg::ROWS + q * 32);
      if (!store) continue;
      if constexpr (MXOUT >= 0) {
        constexpr int kFmt = MXOUT & 1;
        constexpr bool kRowCopy = (MXOUT >> 1) & 1;
        constexpr bool kColCopy = (MXOUT >> 2) & 1;
        constexpr int kEmax = (kFmt == 0) ? 8 : 15;
        const int64_t row = y0 + lane;
        const int64_t col0 = static_cast<int64_t>(nb) * Cfg::BN + half * HALF;
        // both copies are produced chunk by chunk (32 columns at a time), so each chunk's
        // accumulator registers are dead once its codes are out
        uint32_t sbytes = 0;                     // row-wise scale bytes of the 4 chunks
        const int64_t sc_base = (col0 >> 7) * (args.M >> 7) * 512 + (static_cast<int64_t>(y0) >> 7) * 512;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if constexpr (kRowCopy) {
            // row-wise: this thread's row holds the chunk's whole 1x32 block: amax, E8M0 byte
            // max(exp(amax) - emax, 0) (0xFF with codes 0x7F for Inf / NaN), codes of x * 2^-k
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) m = max(m, r[c][i] & 0x7FFFFFFFu);
            uint32_t sb, w[8];
            if (m >= 0x7F800000u) {
              sb = 0xFF;
#pragma unroll
              for (int k = 0; k < 8; ++k) w[k] = 0x7F7F7F7Fu;
            } else {
              const int e = static_cast<int>(m >> 23);
              sb = e > kEmax ? static_cast<uint32_t>(e - kEmax) : 0u;
              const float inv = __uint_as_float((254u - sb) << 23);  // 2^-(sb - 127), always normal
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float f0 = __fmul_rn(__uint_as_float(r[c][4 * k]), inv);
                const float f1 = __fmul_rn(__uint_as_float(r[c][4 * k + 1]), inv);
                const float f2 = __fmul_rn(__uint_as_float(r[c][4 * k + 2]), inv);
                const float f3 = __fmul_rn(__uint_as_float(r[c][4 * k + 3]), inv);
                w[k] = (kFmt == 0) ? (cvt_e4m3x2(f0, f1) | (cvt_e4m3x2(f2, f3) << 16))
                                   : (cvt_e5m2x2(f0, f1) | (cvt_e5m2x2(f2, f3) << 16));
              }
            }
            uint4* dst = reinterpret_cast<uint4*>(args.q_out + row * args.ldc + col0 + c * 32);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            sbytes |= sb << (8 * c);
          }
          if constexpr (kColCopy) {
            // column-wise: the warp's 32 lanes are the 32 rows of one 32x1 block of every column,
            // so a block's amax is one warp reduction; lane l writes row l's code of each column
            // into the transposed copy (32 consecutive bytes per column) and lane i the scale byte
            // of column i, at (column, 32-row block y0 / 32) of the [N][M/32] scales
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint32_t m0 = __reduce_max_sync(0xFFFFFFFFu, r[c][i] & 0x7FFFFFFFu);
              const uint32_t m1 = __reduce_max_sync(0xFFFFFFFFu, r[c][i + 1] & 0x7FFFFFFFu);
              uint32_t sb0 = 0xFF, sb1 = 0xFF;
              float f0 = 0.0f, f1 = 0.0f;
              if (m0 < 0x7F800000u) {
                const int e = static_cast<int>(m0 >> 23);
                sb0 = e > kEmax ? static_cast<uint32_t>(e - kEmax) : 0u;
                f0 = __fmul_rn(__uint_as_float(r[c][i]), __uint_as_float((254u - sb0) << 23));
              }
              if (m1 < 0x7F800000u) {
                const int e = static_cast<int>(m1 >> 23);
                sb1 = e > kEmax ? static_cast<uint32_t>(e - kEmax) : 0u;
                f1 = __fmul_rn(__uint_as_float(r[c][i + 1]), __uint_as_float((254u - sb1) << 23));
              }
              uint32_t w = (kFmt == 0) ? cvt_e4m3x2(f0, f1) : cvt_e5m2x2(f0, f1);
              if (sb0 == 0xFF) w = (w & 0xFF00u) | 0x7Fu;
              if (sb1 == 0xFF) w = (w & 0x00FFu) | 0x7F00u;
              const int64_t col = col0 + c * 32 + i;
              args.q_col[col * args.ldq_col + y0 + lane] = static_cast<uint8_t>(w & 0xFFu);
              args.q_col[(col + 1) * args.ldq_col + y0 + lane] = static_cast<uint8_t>(w >> 8);
              if (lane == i) {
                const int ci = static_cast<int>(col & 127);
                args.s_col[sc_base + chunk_offset_mx(ci) + q] = static_cast<uint8_t>(sb0);
                args.s_col[sc_base + chunk_offset_mx(ci + 1) + q] = static_cast<uint8_t>(sb1);
              }
            }
          }
        }
        if constexpr (kRowCopy) {
          // chunk (row / 128, 128-column block of this half) of the [M][N/32] scales
          *reinterpret_cast<uint32_t*>(args.s_out + ((row >> 7) * (args.N >> 7) + (col0 >> 7)) * 512 +
                                       chunk_offset_mx(static_cast<int>(row & 127))) = sbytes;
        }
      } else {
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        // FP32 output: the chunks of a tile leave spaced out over the next tile's main loop
        // (30 ns per k-step of the tile between chunks, about a quarter of the tile's time in
        // all) instead of in one burst from every SM at once; the bursts slowed the operand
        // loads.  Measured at 8192^3: NVFP4 195.6 -> 191.1 us, MXFP4 180.1 -> 176.7 us, MXFP8
        // (K = 4096) 307.1 -> 302.9 us; bf16 output gained nothing and is not spaced, nor is a
        // CTA's last tile (no main loop follows it).
        if (!OUT_BF16 && c > 0 && tile + nclusters < num_tiles) __nanosleep(static_cast<unsigned>(num_kt) * 30u);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          v[i] = (KIND == kNvf4) ? __fmul_rn(__uint_as_float(r[c][i]), gscale) : __uint_as_float(r[c][i]);
        store_chunk_32x32<OUT_BF16>(&tmOut, buf, v, lane, static_cast<int32_t>(nb * Cfg::BN + half * HALF + c * 32), y0);
      }
      }
    }
  }

  // the output stores complete before the CTA (and its staging buffers) goes away
  if (warp >= 2 && warp < 2 + Cfg::NUM_EPI_WARPS && lane == 0) bulk_wait_all();
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// DeepSeek FP8 GEMM on the CTA pair ("Why FP8 training is stable" (magicnetworld.com), sec 6.3):
// 256 x 256 output tiles, 128 rows per CTA.  Every 128-wide k-block is one TMA stage and four
// kind::f8f6f4 MMAs (M = 256, N = 256: each SM multiplies 128 x 256 per instruction, so every
// operand byte it reads from shared memory feeds twice the work of a 128 x 128 tile) into one of
// two 256-column TMEM buffers, which fill all 512 columns.  The epilogue warps keep the tile's FP32 accumulators in registers (each warp
// 32 rows x 128 columns, i.e. one 128-column weight block, so one scale pair per k-block) and
// promote every k-block as acc += sA[kb][m] * sB[n/128][kb] * P: they read P from TMEM in
// 16-column pieces, the next piece's load overlapping the current piece's paired FMAs, and hand
// the buffer back right after the last piece landed, while the tensor core fills the other one.
// (Measured: 32-column pieces with registers moved from the control warps to the epilogue by
// setmaxnreg ran 12% slower at 4096 x 2048 x 7168.)
// ---------------------------------------------------------------------------------------------
template <bool OUT_BF16, bool GROUPED_ = false>
struct Ds2Cfg {
  static constexpr int BM = 256;
  static constexpr int BN = 256;
  static constexpr int ROWS = 128;     // A rows and B rows each CTA loads
  static constexpr int KBYTES = 128;   // one k-block of E4M3 codes per stage
  static constexpr int A_BYTES = ROWS * KBYTES;
  static constexpr int B_BYTES = ROWS * KBYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int CHUNK_BYTES = OUT_BF16 ? 2048 : 4096;
  static constexpr int STAGING = 8 * CHUNK_BYTES + 1024;
  static constexpr int STATIC_SMEM = GROUPED_ ? (kMaxGroups + 1) * 4 + 64 : 64;  // group table
  static constexpr int STAGES_RAW = (kSmemLimit - 1024 - BAR_BYTES - STAGING - STATIC_SMEM) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING + BAR_BYTES;
  static constexpr int NUM_MMA = KBYTES / 32;
  static constexpr int NBUF = 2;
  static constexpr int BUF_COLS = BN;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_EPI_WARPS = 8;
  static constexpr int EPI_WARP = 2;  // warp 0: producer, warp 1: MMA issuer, 2-9: epilogue
  static constexpr int THREADS = 32 * (EPI_WARP + NUM_EPI_WARPS);
  static_assert(STAGES >= 2, "not enough shared memory");
  static_assert(NBUF * BUF_COLS <= TMEM_COLS, "TMEM overflow");
};

// GROUPED: the DeepSeek expert products of a mixture-of-experts layer in one launch (as for the
// block-scaled kernel: rows off[g] .. off[g+1] of A times the g-th [N][K] block of B, whose
// 128x128 block scales are rows g N / 128 .. of sB; a CTA whose 128 rows lie past its group's
// last row computes but stores nothing).
template <bool OUT_BF16, bool GROUPED = false>
__global__ void __launch_bounds__(Ds2Cfg<OUT_BF16, GROUPED>::THREADS, 1)
    ds_gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
  using Cfg = Ds2Cfg<OUT_BF16, GROUPED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + Cfg::STAGES * Cfg::A_BYTES;
  uint8_t* sOut = sB + Cfg::STAGES * Cfg::B_BYTES;  // 1 KB aligned: stages are multiples of 1 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + Cfg::STAGING);
  uint64_t* full_bar = bars;                       // [STAGES], used in the leader
  uint64_t* empty_bar = bars + Cfg::STAGES;        // [STAGES], both CTAs
  uint64_t* tfull_bar = bars + 2 * Cfg::STAGES;    // [NBUF], both CTAs
  uint64_t* tempty_bar = tfull_bar + Cfg::NBUF;    // [NBUF], used in the leader
  uint64_t* drain_bar = tempty_bar + Cfg::NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int num_mb = args.M / Cfg::BM;
  const int num_nb = args.N / Cfg::BN;
  const int num_kt = args.K / 128;
  __shared__ int grp_start[GROUPED ? kMaxGroups + 1 : 1];  // first tile of each group
  if (GROUPED && threadIdx.x == 0) build_group_table(grp_start, args, Cfg::BM, num_nb);
  // tile -> first A row of the pair, first B row (of the stacked experts), rows of the group from
  // a_row0 on, n-block
  auto decode = [&](int tile, int64_t& a_row0, int64_t& b_row0, int& rows_valid, int& nb) {
    if (GROUPED) {
      int grp;
      decode_group_tile(grp_start, args, Cfg::BM, Cfg::BN, num_nb, tile, grp, a_row0, b_row0, rows_valid, nb);
    } else {
      int mb;
      tile_coords(tile, num_mb, num_nb, mb, nb);
      a_row0 = static_cast<int64_t>(mb) * Cfg::BM;
      b_row0 = static_cast<int64_t>(nb) * Cfg::BN;
      rows_valid = Cfg::BM;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < Cfg::NBUF; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 2 * Cfg::NUM_EPI_WARPS);  // one arrival per epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = GROUPED ? grp_start[args.groups] : num_mb * num_nb;
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
        int64_t a_row0, b_row0;
        int rows_valid, nb;
        decode(tile, a_row0, b_row0, rows_valid, nb);
        const int a_row = static_cast<int>(a_row0) + static_cast<int>(rank) * Cfg::ROWS;
        const int b_row = static_cast<int>(b_row0) + static_cast<int>(rank) * Cfg::ROWS;
        for (int kt = 0; kt < num_kt; ++kt) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = map_to_rank(smem_u32(&full_bar[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * Cfg::STAGE_BYTES);
          tma_load_2d_pair(sA + stage * Cfg::A_BYTES, &tmA, full_leader, kt * Cfg::KBYTES, a_row);
          tma_load_2d_pair(sB + stage * Cfg::B_BYTES, &tmB, full_leader, kt * Cfg::KBYTES, b_row);
          ++issued;
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: the leader's stage barriers count both CTAs' bytes, so the leader waits for every
      // copy either CTA issued; the final cluster barrier keeps the peer alive until then
      if (leader) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
          if (issued > s) {
            const long last = s + ((issued - 1 - s) / Cfg::STAGES) * Cfg::STAGES;
            mbar_wait(&full_bar[s], static_cast<uint32_t>((last / Cfg::STAGES) & 1), abort_flag, kSiteDrain);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      constexpr uint32_t kOpHi = smem_desc_hi(1024, kSwizzle128B);
      constexpr uint32_t kLbo = smem_desc_lo_lbo(16);
      const uint32_t a_lo0 = (smem_u32(sA) >> 4) | kLbo, b_lo0 = (smem_u32(sB) >> 4) | kLbo;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_it = 0;  // k-block partial products handed over so far
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
        for (int kt = 0; kt < num_kt; ++kt) {
          const uint32_t b = acc_it & 1;
          if (!mbar_wait(&tempty_bar[b], ((acc_it >> 1) & 1) ^ 1, abort_flag, kSiteMmaTmemEmpty) ||
              !mbar_wait(&full_bar[stage], phase, abort_flag, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_lo = a_lo0 + stage * (Cfg::A_BYTES >> 4);
          const uint32_t b_lo = b_lo0 + stage * (Cfg::B_BYTES >> 4);
          const uint32_t d_tmem = tmem_base + b * Cfg::BUF_COLS;
#pragma unroll
          for (int j = 0; j < Cfg::NUM_MMA; ++j)
            umma_f8f6f4_pair(d_tmem, desc_from_words(a_lo + j * 2, kOpHi), desc_from_words(b_lo + j * 2, kOpHi),
                             args.idesc, j > 0 ? 1u : 0u);
          umma_commit_pair(&empty_bar[stage], 0x3);
          umma_commit_pair(&tfull_bar[b], 0x3);  // one k-block ready for promotion in both CTAs
          ++acc_it;
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      umma_commit_pair(drain_bar, 0x1);
      mbar_wait(drain_bar, 0, abort_flag, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------------ promotion epilogue
    const int q = warp & 3;                       // TMEM lane quarter
    const int half = (warp - Cfg::EPI_WARP) >> 2;  // which 128-column weight block of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tempty_leader0 = map_to_rank(smem_u32(&tempty_bar[0]), 0);
    const int64_t kbs = num_kt;
    uint8_t* buf = sOut + (warp - Cfg::EPI_WARP) * Cfg::CHUNK_BYTES;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
      int64_t a_row0, b_row0;
      int rows_valid, nb;
      decode(tile, a_row0, b_row0, rows_valid, nb);
      const bool store = static_cast<int>(rank) * Cfg::ROWS < rows_valid;  // this CTA's rows exist
      const int32_t row0 = static_cast<int32_t>(a_row0) + static_cast<int32_t>(rank) * Cfg::ROWS + q * 32;
      // (rows past M, in a grouped tile's unused half, read row M - 1's scales: never stored)
      const int64_t srow = row0 + lane < args.M ? row0 + lane : args.M - 1;
      const float* sa_row = args.dsa + srow;
      const float* sb_blk = args.dsb + (b_row0 / 128 + half) * kbs;
      float nsa = __ldg(sa_row), nsb = __ldg(sb_blk);
      uint64_t acc[64];  // this thread's 128 FP32 accumulators as pairs
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0ull;
      for (int kt = 0; kt < num_kt; ++kt) {
        const float s = __fmul_rn(nsa, nsb);
        if (kt + 1 < num_kt) {
          nsa = __ldg(sa_row + static_cast<int64_t>(kt + 1) * args.M);
          nsb = __ldg(sb_blk + kt + 1);
        }
        const uint32_t b = acc_it & 1;
        ok = mbar_wait(&tfull_bar[b], (acc_it >> 1) & 1, abort_flag, kSiteEpiTmemFull);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + b * Cfg::BUF_COLS + half * 128;
        const uint64_t s2 = pack_f32x2(s, s);
        uint32_t r[2][16];
        tmem_ld_32x32b_x16(taddr, r[0]);
        tmem_ld_wait();
        tmem_regs_ready16(r[0]);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c < 7) tmem_ld_32x32b_x16(taddr + (c + 1) * 16, r[(c + 1) & 1]);
#pragma unroll
          for (int i = 0; i < 8; ++i) fma2_scalar(acc[c * 8 + i], s2, r[c & 1][2 * i], r[c & 1][2 * i + 1]);
          if (c < 7) {
            tmem_ld_wait();
            tmem_regs_ready16(r[(c + 1) & 1]);
          }
          if (c == 6) {
            // every piece of P is in registers: hand the buffer back before the last FMAs
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8 * b);
          }
        }
        ++acc_it;
      }
      if (!ok) break;
      if (!store) continue;
      // the tile's 32 rows x 128 columns, as four 32 x 32 TMA stores through the staging buffer
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) unpack_f32x2(acc[c * 16 + i], v[2 * i], v[2 * i + 1]);
        store_chunk_32x32<OUT_BF16>(&tmOut, buf, v, lane, nb * Cfg::BN + half * 128 + c * 32, row0);
      }
    }
  }

  if (warp >= Cfg::EPI_WARP && lane == 0) bulk_wait_all();
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
}

}  // namespace mxgb
