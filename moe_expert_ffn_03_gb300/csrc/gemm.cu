// Grouped block-scaled MXFP8 GEMM on the sm_103a tensor cores (tcgen05).
//
// Page "Efficient MoE Training for Biological Foundation Models":
//   section "GroupedLinear": all experts' GEMMs are submitted as ONE grouped
//   operation driven by split_sizes instead of one launch per expert;
//   section "MXFP8与融合MLP": MXFP8 GEMMs run on dedicated Blackwell tensor
//   core instructions, and quantization, SwiGLU and the router-probability
//   scaling are fused into the grouped MLP so no intermediate is stored in
//   high precision.
//
// Design (persistent; CTA pairs of a 2-CTA cluster, one CTA per SM):
//   Each pair computes a 256 x 256 output tile with tcgen05.mma.cta_group::2
//   (M = 256): the even CTA of the cluster (the leader) holds rows 0..127 of
//   the tile and the left 128 columns of B, the odd CTA (the peer) rows
//   128..255 and the right 128 columns.  Each SM thus stages 32 KB of operands
//   per 128-deep K step instead of 48 KB for the same tensor work, and the
//   ring has 6 slots (4 for the SwiGLU-backward kinds), filled and released
//   two at a time.
//   warp 0      (both CTAs) TMA producer: per barrier stage (two 128-byte K
//               steps) one 3-D box of the CTA's 128 A rows and one of its 128 B
//               rows (128B swizzle; each lands as two K-step tiles) and, for
//               MXFP8, the scale atoms of its A rows and of all 256 B rows;
//               every copy signals the leader's full barrier of the stage
//               (.cta_group::2), which the leader alone arms with both CTAs'
//               byte count.
//   warp 1      allocates TMEM (collectively with the peer); in the leader it
//               issues, per K step, the scale-factor copies (tcgen05.cp, ordered
//               before the MMAs that read them) and four tcgen05.mma (M=256,
//               N=256, K=32); tcgen05.commit multicasts the stage release to both
//               CTAs and, after the last K step, hands each CTA its half of the
//               accumulator (fp32, 256 columns).  Kinds without scale factors
//               (bf16, per-tensor E4M3) alternate two 256-column accumulators.
//   warps 2..17 (both CTAs) epilogue, four per TMEM lane quarter (32 rows), 64
//               accumulator columns each: tcgen05.ld into registers, release the
//               accumulator at once (an arrival on the leader's barrier), then
//               the fused epilogue math (bf16 store, ScaledSwiGLU +
//               re-quantization along both axes, or SwiGLU backward +
//               re-quantization, its saved g,u staged in shared memory by
//               cp.async ahead of use).
// Tiles: mode 0 walks pairs of 128-row blocks inside each expert segment
// (computed on the device from split_sizes; empty experts get no tile; the
// second block of an expert with an odd block count is computed and dropped)
// times the N tiles, rasterised in groups of 8 pairs; mode 1 (weight
// gradients) walks expert x 256-row M tiles x N tiles with K = the expert's
// padded token range.
// Every mbarrier wait is bounded; on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT, stops issuing, drains its copies and MMAs, frees
// TMEM and returns.
//
// The file also holds the router's weight gradient on the tensor cores
// (router_dw_tc_kernel: single-CTA MMAs on MN-major operands, dl as two bf16
// terms), which shares these PTX wrappers and the bounded waits.
#include <cuda.h>

#include <atomic>
#include <cstdio>

#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;     // BM: rows per CTA; the pair's MMA has M = 2 * BM
constexpr int MMA_M = 2 * BM;
constexpr int A_TILE = BM * BK;                 // 16 KB of E4M3
constexpr int B_HALF = 128 * BK;                // 16 KB: one 128-row box of B (this CTA's half of N)
constexpr int SF_ATOM = 512;                    // 128 rows x 4 scale bytes
constexpr int NUM_EPI_WARPS = 16;               // 4 per TMEM lane quarter
constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_ACC = 0;                  // accumulator: columns 0..255
constexpr uint32_t TM_SF0 = 256, TM_SF_STRIDE = 12;  // per stage: SFA 4 columns + SFB 8 columns
// Columns 384..511: per epilogue warp a 32-column parking place (lanes of its quarter)
// for the second half of its accumulator columns in the SwiGLU-backward epilogue.
constexpr uint32_t TM_STASH = 384;
// MXFP8 SwiGLU backward (four slots, so its scale columns end at 304): per epilogue warp
// 48 columns 304 + 48*cg .. (lanes of its quarter) hold columns 16..63 of its dA; columns
// 0..15 stay in registers.
constexpr uint32_t TM_DA_STASH = 304, TM_DA_STASH_W = 48;
constexpr int GROUP_M = 8;
constexpr int SEG_INTS = 260;                   // per-expert prefix of 128-row blocks (E <= 256, plus the total)
constexpr int kMaxSegE = 256;                   // mode-1 expert order (heaviest first) follows the prefix
constexpr int SEG_PB = SEG_INTS + kMaxSegE;     // then the per-expert prefix of block pairs (mode 0)
constexpr int TR_PITCH = 9;                     // floats per row of a warp's 32x8 transpose buffer
constexpr int TR_WARP_FLOATS = 32 * TR_PITCH;
// g,u staging of the SwiGLU backward: per lane (row) 32 g then 32 u values, eight
// 16-byte chunks in a 128-byte row; chunk c of lane l sits at chunk c ^ (l & 7), so a
// quarter warp reading one chunk index touches eight distinct bank groups.
constexpr int GU_PITCH = 128;

// bf16-operand kinds: 64 K elements per 128-byte stage row, kind::f16 MMA, no scales.
// Per-tensor E4M3 kinds: 128 K elements per stage, kind::f8f6f4 MMA, no block scales.
template <int EPI>
struct Ops {
  static constexpr bool B16 = (EPI == EPI_B16_OUT || EPI == EPI_B16_FWD_SWIGLU || EPI == EPI_B16_BWD_SWIGLU);
  static constexpr bool SWIGLU_BWD = (EPI == EPI_BWD_SWIGLU || EPI == EPI_B16_BWD_SWIGLU || EPI == EPI_T8_BWD_SWIGLU);
  static constexpr bool T8 = (EPI == EPI_T8_OUT || EPI == EPI_T8_FWD_SWIGLU || EPI == EPI_T8_BWD_SWIGLU);
  static constexpr bool NOSF = B16 || T8;         // no scale-factor loads or copies
  static constexpr bool SWIGLU_FWD = (EPI == EPI_FWD_SWIGLU || EPI == EPI_B16_FWD_SWIGLU || EPI == EPI_T8_FWD_SWIGLU);
  static constexpr int KSTEP = B16 ? 64 : 128;    // K elements per stage
  // Kinds without scale factors leave TMEM to the accumulator: two 256-column
  // buffers, so the next tile's MMAs run while the epilogue drains the last one.
  // The SwiGLU-backward kinds park half their columns in TMEM and keep one buffer.
  static constexpr int ACC_BUFS = (NOSF && !SWIGLU_BWD) ? 2 : 1;
};

// Shared-memory layout (per CTA; both CTAs of a pair use the same offsets): six
// slots (four for the SwiGLU-backward kinds, which stage g,u instead), each one
// 128-deep K step of the CTA's A box, its B box and the scale
// atoms (its A rows; the two 128-row blocks of B), then the barriers, the segment
// tables and the epilogue warps' transpose buffers.  The slots are filled and
// released two at a time (one barrier stage = 256 of K, 64 KB of operands):
// measured on this GPU, what TMA delivers to an SM grows with the bytes behind
// each barrier stage (about 35 B/clk with 32 KB stages, 50 with 64 KB), and the
// pair needs 64 B/clk per SM to keep its MMAs busy.
constexpr int STAGE_STEPS = 2;                  // K steps (slots) per barrier stage

template <int EPI>
struct Lay {
  // The SwiGLU-backward kinds, bound by their epilogue, trade two slots for a per-warp
  // staging buffer of the saved g,u (one half of the warp's columns, 32 rows).
  static constexpr int STG = Ops<EPI>::SWIGLU_BWD ? 4 : 6;   // slots of one K step
  static constexpr int PER = STAGE_STEPS;        // slots per barrier stage
  static constexpr int NSTG = STG / PER;         // barrier stages
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STG * A_TILE;
  static constexpr int OFF_SFA = OFF_B + STG * B_HALF;      // per slot: the atom of this CTA's A rows
  static constexpr int OFF_SFB0 = OFF_SFA + STG * SF_ATOM;  // per slot: the atom of B rows 0..127
  static constexpr int OFF_SFB1 = OFF_SFB0 + STG * SF_ATOM; // per slot: the atom of B rows 128..255
  static constexpr int OFF_BAR = OFF_SFB1 + STG * SF_ATOM;
  // full[NSTG] (leader: both CTAs' copies), empty[NSTG], tmem_full[2], tmem_empty[2] (leader:
  // both CTAs' epilogue warps), drain (MMA)
  static constexpr int NUM_BARS = 2 * NSTG + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_SEG = OFF_MISC + 16;             // seg_mb[SEG_INTS], order[kMaxSegE], seg_pb[SEG_INTS]
  static constexpr int OFF_TR = (OFF_SEG + (2 * SEG_INTS + kMaxSegE) * 4 + 15) & ~15;
  static constexpr int OFF_GU = OFF_TR + NUM_EPI_WARPS * TR_WARP_FLOATS * 4;
  static constexpr int GU_WARP = Ops<EPI>::SWIGLU_BWD ? 32 * GU_PITCH : 0;
  static constexpr int SMEM_USED = OFF_GU + NUM_EPI_WARPS * GU_WARP;
  static_assert(OFF_GU % 16 == 0 && GU_PITCH % 16 == 0, "16-byte cp.async and vector reads of the g,u staging");
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 B
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(TM_SF0 + STG * TM_SF_STRIDE <= TM_STASH, "TMEM budget");
  static_assert(EPI != EPI_BWD_SWIGLU ||
                    (TM_SF0 + STG * TM_SF_STRIDE <= TM_DA_STASH && TM_DA_STASH + 4 * TM_DA_STASH_W <= TMEM_COLS),
                "TMEM budget of the dA stash");
  static_assert(STG % PER == 0, "slots come in whole barrier stages");
};

// ---- PTX wrappers -------------------------------------------------------------------
// Cluster helpers.  A shared::cta address of this CTA is also its shared::cluster
// address; mapa gives the address of the same offset in another CTA of the cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier anywhere in the cluster, without release semantics: the arrival
// does not wait for this thread's earlier global stores to be performed.  For handing the
// accumulator back to the MMA warp, which needs only this warp's TMEM reads finished:
// tcgen05.wait::ld has returned (the values are in registers) and
// tcgen05.fence::before_thread_sync orders them before the arrival.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t caddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// Tensor copy into this CTA's shared memory; completion is signalled on the
// mbarrier at cluster address bar_c, which may sit in the pair's other CTA.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint32_t bar_c) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_c)
      : "memory");
}
// 3-D copy: {x in the 128-byte K atom, row, K atom}; a {.., 128, STAGE_STEPS} box lands
// as 128-row SW128 tiles back to back, one per K step of a barrier stage.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint32_t bar_c) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_c)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Arrives, once the pair's earlier tcgen05 operations are done, on the mbarrier at
// this offset in both CTAs of the pair.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      ::"r"(smem_u32(bar)), "h"(uint16_t(3))
      : "memory");
}
// Each CTA of the pair copies the atom at this shared-memory offset into its own TMEM.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i).  The
// registers are valid only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns (valid after tmem_wait_ld).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns (valid after tmem_wait_ld).
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Wait for this thread's outstanding tcgen05.ld; the empty asm statements tie
// every loaded register to the wait so no use is scheduled before it.
template <int N>
__device__ __forceinline__ void tmem_wait_ld(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Shared-memory matrix descriptor, K-major operand staged by TMA with 128-byte
// swizzle: 8-row x 128-byte swizzle atoms stacked every 1024 bytes (SBO);
// the leading-dimension offset is unused for swizzled K-major layouts.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(1) << 16;                 // LBO (ignored), encoded 16 B
  d |= uint64_t(1024 >> 4) << 32;         // SBO
  d |= uint64_t(1) << 46;                 // descriptor version of the sm_100 family
  d |= uint64_t(2) << 61;                 // SWIZZLE_128B
  return d;
}
// Descriptor of one 512-byte scale atom as 32 rows x 16 bytes, no swizzle:
// 8-row core matrices every 128 bytes.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(128 >> 4) << 32;
  d |= uint64_t(1) << 46;
  return d;
}
// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 x E4M3,
// both K-major, UE8M0 scales, scale-factor ids select the byte (= 32-block of
// the 128-deep K step) inside each 32-bit TMEM scale word.
__device__ __forceinline__ uint32_t idesc_mxf8(int N, int sf_id) {
  return (uint32_t(sf_id) << 4)            // B scale factor id
         | (0u << 7) | (0u << 10)          // A, B format E4M3
         | (uint32_t(N >> 3) << 17)        // N / 8
         | (1u << 23)                      // scale format UE8M0
         | (uint32_t(MMA_M >> 4) << 24)    // M / 16
         | (uint32_t(sf_id) << 29);        // A scale factor id
}

// Instruction descriptor of kind::f16: bf16 x bf16 -> f32, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int N) {
  return (1u << 4)                         // D format F32
         | (1u << 7) | (1u << 10)          // A, B format BF16
         | (uint32_t(N >> 3) << 17)        // N / 8
         | (uint32_t(MMA_M >> 4) << 24);   // M / 16
}
// Instruction descriptor of kind::f8f6f4 without block scaling: E4M3 x E4M3 -> f32, both K-major.
__device__ __forceinline__ uint32_t idesc_f8(int N) {
  return (1u << 4)                         // D format F32
         | (0u << 7) | (0u << 10)          // A, B format E4M3
         | (uint32_t(N >> 3) << 17)        // N / 8
         | (uint32_t(MMA_M >> 4) << 24);   // M / 16
}
__device__ __forceinline__ void tc_mma_f8(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One CTA's view of a pair tile.
struct Tile {
  int e;
  int nb;
  int k_tiles;
  int n0;
  bool second;            // output columns n0+128.. of the tile exist (or the up half of a ScaledSwiGLU tile)
  bool valid;             // this CTA's 128 rows belong to the tile (the peer's half can fall past the expert)
  int64_t a_row;          // this CTA's first row of A
  int64_t k0;             // first K element
  int64_t b_row0, b_row1; // rows of B: the leader's half (columns 0..127) and the peer's (128..255)
  int64_t out_row;        // output row of this CTA's row 0 (mode 1: e*M + a_row)
};

__device__ __forceinline__ int tile_count(const GemmArgs& a, const int* seg) {
  if (a.mode == 0) return seg[SEG_PB + a.E] * a.n_tiles;
  return a.E * ((a.M + MMA_M - 1) / MMA_M) * a.n_tiles;
}

// seg: prefix of 128-row blocks per expert [0..E], the mode-1 expert order at
// SEG_INTS, the prefix of block pairs per expert at SEG_PB.  rank: 0 (leader) or 1.
template <int EPI>
__device__ __forceinline__ void decode_tile(const GemmArgs& a, const int* seg, int t, int rank, Tile& tl) {
  if (a.mode == 0) {
    const int* seg_pb = seg + SEG_PB;
    const int total_pb = seg_pb[a.E];
    const int per_group = GROUP_M * a.n_tiles;
    const int group = t / per_group;
    const int first = group * GROUP_M;
    const int gs = min(GROUP_M, total_pb - first);
    const int local = t - group * per_group;
    const int pb = first + local % gs;
    const int nb = local / gs;
    int lo = 0, hi = a.E - 1;            // largest e with seg_pb[e] <= pb
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg_pb[mid] <= pb) lo = mid; else hi = mid - 1;
    }
    const int blk = 2 * (pb - seg_pb[lo]) + rank;    // 128-row block inside the expert's segment
    tl.e = lo;
    tl.nb = nb;
    tl.valid = blk < seg[lo + 1] - seg[lo];
    tl.a_row = int64_t(seg[lo] + blk) * BM;
    tl.k0 = 0;
    tl.k_tiles = a.K / Ops<EPI>::KSTEP;
    tl.out_row = tl.a_row;
    if (Ops<EPI>::SWIGLU_FWD) {
      tl.n0 = nb * 128;
      tl.b_row0 = int64_t(lo) * a.b_rows_per_expert + tl.n0;
      tl.b_row1 = tl.b_row0 + a.I;
      tl.second = true;
    } else {
      tl.n0 = nb * BN;
      tl.b_row0 = int64_t(lo) * a.b_rows_per_expert + tl.n0;
      tl.b_row1 = tl.b_row0 + 128;
      tl.second = (tl.n0 + 128) < a.N;
    }
  } else {
    // experts in order of decreasing token count (seg is followed by that order), so the
    // longest tiles are spread over the pairs first and the short ones fill in at the end
    const int m_tiles = (a.M + MMA_M - 1) / MMA_M;
    const int per_e = m_tiles * a.n_tiles;
    const int slot = t / per_e;
    const int e = seg[SEG_INTS + slot];
    const int rem = t - slot * per_e;
    const int mb = rem / a.n_tiles;
    const int nb = rem - mb * a.n_tiles;
    tl.e = e;
    tl.nb = nb;
    tl.a_row = int64_t(mb) * MMA_M + rank * BM;
    tl.valid = tl.a_row < a.M;
    tl.k0 = int64_t(seg[e]) * 128;
    tl.k_tiles = (seg[e + 1] - seg[e]) * (128 / Ops<EPI>::KSTEP);
    tl.n0 = nb * BN;
    tl.b_row0 = tl.n0;
    tl.b_row1 = tl.n0 + 128;
    tl.second = (tl.n0 + 128) < a.N;
    tl.out_row = int64_t(e) * a.M + tl.a_row;
  }
}

// Global sources of one CTA's K steps: TMA coordinates of its A and B boxes and
// the rows (in 256-byte units, two per atom) of the scale atoms it stages.
struct TileSrc {
  int e;
  int a_row, b_row, k0, k_tiles;
  int sfa_y, sfb0_y, sfb1_y;
};

template <int EPI>
__device__ __forceinline__ void tile_src(const GemmArgs& a, const int* seg, int t, int rank, TileSrc& ts) {
  Tile tl;
  decode_tile<EPI>(a, seg, t, rank, tl);
  const int64_t sfa_row_atoms = a.sfa_K / BK;
  const int64_t sfb_row_atoms = a.sfb_K / BK;
  ts.e = tl.e;
  ts.a_row = int(tl.a_row);
  ts.b_row = int(rank == 0 ? tl.b_row0 : tl.b_row1);
  ts.k0 = int(tl.k0);
  ts.k_tiles = tl.k_tiles;
  ts.sfa_y = int(2 * ((tl.a_row / BM) * sfa_row_atoms + tl.k0 / BK));
  ts.sfb0_y = int(2 * ((tl.b_row0 / 128) * sfb_row_atoms + tl.k0 / BK));
  ts.sfb1_y = int(2 * ((tl.b_row1 / 128) * sfb_row_atoms + tl.k0 / BK));
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA aborted or
// the limit ran out (then records the timeout and raises the abort flag).
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                        int site, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        report_error(err, MOE_ERR_DEVICE_TIMEOUT, site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---- epilogues ---------------------------------------------------------------------
// 32 floats of one row as bf16 (64 bytes at p): two 256-bit stores when the output's base
// pointers are 32-byte aligned (v8, set by the host; the offsets are multiples of 64
// bytes), else four 16-byte stores.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, const float* v, bool v8) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[16 * h + 2 * i], v[16 * h + 2 * i + 1]);
    if (v8) {
      st_global_v8(p + 16 * h, w);
    } else {
      uint4* p4 = reinterpret_cast<uint4*>(p + 16 * h);
      p4[0] = make_uint4(w[0], w[1], w[2], w[3]);
      p4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// ---- MX quantization pieces of the epilogues --------------------------------------
// Block maximum of |v| raised by two values, as a float: non-negative floats order like
// their bits, so this is the integer maximum of the |v| bit patterns for finite values;
// max.NaN propagates a NaN, and a NaN or Inf maximum has exponent field 255, which
// mx_scale_code turns into the NaN scale -- the same code as the integer form gives.
__device__ __forceinline__ float amax_raise(float m, float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
  return r;
}

// Eight values of a block whose scale code c is known -> eight E4M3 codes (two words,
// value 0 in the low byte of the first): v * 2^(127 - c) rounded to nearest even, or the
// NaN codes when c is the NaN scale.
__device__ __forceinline__ uint2 mx_encode8(const float* v, uint32_t c) {
  if (c == 255u) return make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const float m = mx_inv_scale(c);
  const float2 m2 = make_float2(m, m);
  const float2 a = __fmul2_rn(make_float2(v[0], v[1]), m2), b = __fmul2_rn(make_float2(v[2], v[3]), m2);
  const float2 e = __fmul2_rn(make_float2(v[4], v[5]), m2), f = __fmul2_rn(make_float2(v[6], v[7]), m2);
  return make_uint2(cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16),
                    cvt_e4m3x2(e.x, e.y) | (cvt_e4m3x2(f.x, f.y) << 16));
}

// Keeps a pointer opaque to the compiler, so that an unrolled loop advances it step by step
// instead of holding every step's precomputed address in registers.
__device__ __forceinline__ void opaque(uint8_t*& p) { asm volatile("" : "+l"(p)); }


// Along-token quantization: where lane (c = lane/4, g = lane%4) of a warp whose 32 lanes
// are the rows row_blk0.. writes the codes of column col + c (rows 8g..8g+7 of its block)
// and that column's scale, in the transposed [cols][cap] tensor.  The next eight columns
// (the next round) are 8*cap bytes further for the codes and 128 bytes further for the
// scale: col is a multiple of 32, so the rounds stay inside one 32-row group of the scale
// atom.
struct ColDst {
  uint8_t* codes;
  uint8_t* scales;
};
__device__ __forceinline__ ColDst col_dst(uint8_t* codes_t, uint8_t* scales_t, int64_t row_blk0, int64_t col,
                                          int64_t cap, int lane) {
  const int64_t crow = col + (lane >> 2);
  return ColDst{codes_t + crow * cap + row_blk0 + 8 * (lane & 3), scales_t + sf_offset(crow, row_blk0 >> 5, cap)};
}

// One round of the along-token quantizer: eight columns of the warp's 32 consecutive
// permuted rows (one MX block along tokens; lane = row, v = this lane's eight values).
// The eight columns go through the warp's shared-memory buffer (32 rows x 9 floats,
// conflict-free both ways): lane (c = lane/4, g = lane%4) then holds rows 8g..8g+7 of
// column c, takes the block maximum with two shuffles and stores its 8 codes as one
// 8-byte word at dst.codes; the g == 0 lane stores the column's scale at dst.scales.
__device__ __forceinline__ void quant_col_round(const float* v, ColDst dst, int lane, float* tr) {
  const int c = lane >> 2, g = lane & 3;
#pragma unroll
  for (int t = 0; t < 8; ++t) tr[lane * TR_PITCH + t] = v[t];
  __syncwarp();
  float w[8];
  float amax = 0.f;
#pragma unroll
  for (int t = 0; t < 8; ++t) w[t] = tr[(8 * g + t) * TR_PITCH + c];
  __syncwarp();
#pragma unroll
  for (int t = 0; t < 8; t += 2) amax = amax_raise(amax, w[t], w[t + 1]);
  uint32_t ab = __float_as_uint(amax);
  ab = max(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 1));
  ab = max(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 2));
  const uint32_t sc = mx_scale_code(ab);
  *reinterpret_cast<uint2*>(dst.codes) = mx_encode8(w, sc);
  if (g == 0) *dst.scales = uint8_t(sc);
}
__device__ __forceinline__ void next_round(ColDst& d, int64_t cap) {
  d.codes += 8 * cap;
  d.scales += 128;
  opaque(d.codes);
  opaque(d.scales);
}

// 32 values of one column block (this thread's row) quantized rowwise; the scale
// of (row, block) goes to the tile layout with row length K.
__device__ __forceinline__ void quant_row_block(const float* v, uint8_t* codes, uint8_t* scales, int64_t row,
                                                int64_t col, int64_t K) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 2) amax = amax_raise(amax, v[i], v[i + 1]);
  const uint32_t c = mx_scale_code(__float_as_uint(amax));
  uint32_t q[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint2 e = mx_encode8(v + 8 * j, c);
    q[2 * j] = e.x;
    q[2 * j + 1] = e.y;
  }
  st_global_v8(codes + row * K + col, q);
  scales[sf_offset(row, col >> 5, K)] = uint8_t(c);
}

// The same 32 columns quantized along tokens: four rounds of eight columns.
__device__ __forceinline__ void quant_col_block(const float* v, uint8_t* codes_t, uint8_t* scales_t,
                                                int64_t row_blk0, int64_t col, int64_t cap, int lane,
                                                float* tr) {
  ColDst d = col_dst(codes_t, scales_t, row_blk0, col, cap, lane);
#pragma unroll
  for (int rnd = 0; rnd < 4; ++rnd) {
    quant_col_round(v + 8 * rnd, d, lane, tr);
    next_round(d, cap);
  }
}

// ScaledSwiGLU backward of two columns of one row (a = silu(g)*u*p): with s = sigmoid(g)
// and dp = dA*p,
//   dg = dp*u*s*(1 + g*(1 - s)),  du = dp*g*s,  and sg*u = g*s*u for the row sum of dA*silu(g)*u.
// Packed float32x2 arithmetic; exp and the reciprocal are the hardware approximations
// (about 2 ulp; the results feed E4M3 quantizers with 3 mantissa bits).
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// ScaledSwiGLU of two columns: a = silu(g) * u * p with silu(g) = g / (1 + e^-g), the
// quotient as g times the approximate reciprocal (the result feeds an E4M3 quantizer).
__device__ __forceinline__ float2 scaled_swiglu2(float2 g, float2 u, float2 p2) {
  const float2 t = __fmul2_rn(g, make_float2(-1.4426950408889634f, -1.4426950408889634f));   // -g log2(e)
  const float2 den = __fadd2_rn(make_float2(1.f, 1.f), make_float2(ex2_approx(t.x), ex2_approx(t.y)));
  const float2 sg = __fmul2_rn(g, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
  return __fmul2_rn(__fmul2_rn(sg, u), p2);
}
__device__ __forceinline__ void swiglu_bwd2(float2 d, float2 g, float2 u, float2 p2, float2& dg, float2& du,
                                            float2& sgu) {
  const float2 one = make_float2(1.f, 1.f);
  const float2 t = __fmul2_rn(g, make_float2(-1.4426950408889634f, -1.4426950408889634f));   // -g log2(e)
  const float2 den = __fadd2_rn(one, make_float2(ex2_approx(t.x), ex2_approx(t.y)));          // 1 + e^-g
  const float2 s = make_float2(rcp_approx(den.x), rcp_approx(den.y));
  const float2 sg = __fmul2_rn(g, s);
  const float2 oms = __ffma2_rn(s, make_float2(-1.f, -1.f), one);                              // 1 - s
  const float2 dsilu = __fmul2_rn(s, __ffma2_rn(g, oms, one));
  const float2 dpa = __fmul2_rn(d, p2);
  dg = __fmul2_rn(__fmul2_rn(dpa, u), dsilu);
  du = __fmul2_rn(dpa, sg);
  sgu = __fmul2_rn(sg, u);
}

// SiLU with the fast divide (__fdividef, about 2 ulp): the result feeds an E4M3
// quantizer (3 mantissa bits) or a bf16 store.  For g below about -87 the
// denominator passes 2^126 and it returns 0 (the exact value there is below
// 1e-35 in magnitude).
// The same 32 columns stored transposed as bf16 (the bf16 path's along-token copy):
// column col+i becomes row col+i of [cols][cap]; through the warp's transpose
// buffer eight columns at a time, lane (c = lane/4, g = lane%4) writes rows
// 8g..8g+7 of column c as one 16-byte store.
__device__ __forceinline__ void store_col_bf16(const float* v, __nv_bfloat16* out_t, int64_t row_blk0, int64_t col,
                                               int64_t cap, int lane, float* tr) {
  const int c = lane >> 2, g = lane & 3;
#pragma unroll
  for (int rnd = 0; rnd < 4; ++rnd) {
#pragma unroll
    for (int t = 0; t < 8; ++t) tr[lane * TR_PITCH + t] = v[8 * rnd + t];
    __syncwarp();
    float w[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) w[t] = tr[(8 * g + t) * TR_PITCH + c];
    __syncwarp();
    const int64_t crow = col + 8 * rnd + c;
    *reinterpret_cast<uint4*>(out_t + crow * cap + row_blk0 + 8 * g) =
        make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
  }
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// One epilogue warp on one tile.  The warp owns TMEM lane quarter q (32 rows) and
// column group cg: 64 accumulator columns cg*64.. of an N=256 tile, or gate
// columns cg*32.. and up columns 128+cg*32.. of a ScaledSwiGLU tile.  It pulls its
// columns into registers, releases the accumulator (an arrival on the leader's
// tmem_empty, at cluster address tmem_empty_c) and only then runs the epilogue
// math, so the next tile's MMAs overlap it.  A CTA whose half of the pair tile
// lies past the expert's rows (or past M) releases the accumulator and writes nothing.
// This lane's saved g and u (32 columns each from col) into its row of the warp's
// staging buffer; completes with cp_async_wait_all.
__device__ __forceinline__ void stage_gu(const GemmArgs& a, int64_t row, int64_t col, uint8_t* gu_s, int sw) {
  const __nv_bfloat16* grow = a.gu + row * (2 * int64_t(a.I)) + col;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    cp_async16(gu_s + ((j ^ sw) << 4), grow + 8 * j, true);
    cp_async16(gu_s + (((4 + j) ^ sw) << 4), grow + a.I + 8 * j, true);
  }
}

// dA of chunk j of half h of an epilogue warp's 64 columns: columns 0..15 are in registers
// r, columns 16..63 in the warp's TMEM stash.  da_issue starts the chunk's load (a copy for
// the register chunks); da_land waits for it, so the load can run under other work.
__device__ __forceinline__ void da_issue(const uint32_t* r, uint32_t stash, int h, int j, uint32_t* d) {
  if (h == 0 && j < 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = r[8 * j + i];
  } else {
    tmem_ld8_async(stash + uint32_t(8 * (4 * h + j - 2)), d);
  }
}
__device__ __forceinline__ void da_land(int h, int j, uint32_t* d) {
  if (!(h == 0 && j < 2)) tmem_wait_ld<8>(d);
}

// Chunk j (columns 8j..8j+7 of the half starting at col) of this lane's g and u into its
// row of the staging buffer; completes with cp_async_wait_all.
__device__ __forceinline__ void stage_gu_chunk(const GemmArgs& a, int64_t row, int64_t col, uint8_t* gu_s, int sw,
                                               int j) {
  const __nv_bfloat16* grow = a.gu + row * (2 * int64_t(a.I)) + col;
  cp_async16(gu_s + ((j ^ sw) << 4), grow + 8 * j, true);
  cp_async16(gu_s + (((4 + j) ^ sw) << 4), grow + a.I + 8 * j, true);
}

// dg and du of chunk j (eight columns) of this lane's row from its dA (d[0..7]), its
// staged g,u and p; with dp2 != nullptr the chunk's dA*silu(g)*u is added to the pair sum.
__device__ __forceinline__ void swiglu_bwd_chunk(const uint32_t* d, const uint8_t* gu_s, int j, int lane,
                                                 float2 p2, float* vg, float* vu, float2* dp2) {
  const uint4 gw = *reinterpret_cast<const uint4*>(gu_s + ((j ^ (lane & 7)) << 4));
  const uint4 uw = *reinterpret_cast<const uint4*>(gu_s + (((4 + j) ^ (lane & 7)) << 4));
  const uint32_t gs[4] = {gw.x, gw.y, gw.z, gw.w};
  const uint32_t us[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float2 dg, du, sgu;
    const float2 dd = make_float2(__uint_as_float(d[2 * t]), __uint_as_float(d[2 * t + 1]));
    swiglu_bwd2(dd, make_float2(bf16_lo(gs[t]), bf16_hi(gs[t])), make_float2(bf16_lo(us[t]), bf16_hi(us[t])), p2,
                dg, du, sgu);
    if (dp2 != nullptr) *dp2 = __ffma2_rn(dd, sgu, *dp2);
    vg[2 * t] = dg.x;
    vg[2 * t + 1] = dg.y;
    vu[2 * t] = du.x;
    vu[2 * t + 1] = du.y;
  }
}

template <int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, const Tile& tl, uint32_t tmem_row, int q, int cg,
                                              int lane, uint32_t tmem_empty_c, float* tr, uint8_t* gu_s) {
  if (!tl.valid) {
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster_relaxed(tmem_empty_c);
    return;
  }
  const int64_t row = tl.out_row + q * 32 + lane;        // output / permuted row of this thread
  const int64_t row_blk0 = tl.out_row + q * 32;
  const int ncols = tl.second ? 256 : 128;                // valid accumulator columns
  const int c0 = cg * 64;
  uint32_t r[64];
  bool have;
  if (Ops<EPI>::SWIGLU_FWD) {
    have = true;
    tmem_ld32_async(tmem_row + TM_ACC + cg * 32, r);
    tmem_ld32_async(tmem_row + TM_ACC + 128 + cg * 32, r + 32);
    tmem_wait_ld<64>(r);
  } else if (EPI == EPI_BWD_SWIGLU) {
    // columns 16..63 of this warp's dA go to its TMEM stash (32 and 16 columns), columns
    // 0..15 stay in registers; then the accumulator is free for the next tile
    have = c0 < ncols;
    if (have) {
      // two TMEM round trips before the accumulator is released (it gates the next tile's MMAs)
      const uint32_t stash = tmem_row + TM_DA_STASH + uint32_t(cg) * TM_DA_STASH_W;
      tmem_ld32_async(tmem_row + TM_ACC + c0 + 16, r);
      tmem_ld16_async(tmem_row + TM_ACC + c0 + 48, r + 32);
      tmem_wait_ld<48>(r);
      tmem_st32(stash, r);
      tmem_st16(stash + 32, r + 32);
      tmem_ld16_async(tmem_row + TM_ACC + c0, r);
      tmem_wait_ld<16>(r);
      tmem_wait_st();
    }
  } else if (Ops<EPI>::SWIGLU_BWD) {
    // 64 columns do not fit the register budget next to the SwiGLU-backward math:
    // park the second 32 in this warp's spare TMEM columns, then free the accumulator
    have = c0 < ncols;
    if (have) {
      tmem_ld32_async(tmem_row + TM_ACC + c0 + 32, r);
      tmem_wait_ld<32>(r);
      tmem_st32(tmem_row + TM_STASH + cg * 32, r);
      tmem_ld32_async(tmem_row + TM_ACC + c0, r);
      tmem_wait_ld<32>(r);
      tmem_wait_st();
    }
  } else {
    have = c0 < ncols && tl.k_tiles > 0;
    if (have) {
      tmem_ld32_async(tmem_row + TM_ACC + c0, r);
      tmem_ld32_async(tmem_row + TM_ACC + c0 + 32, r + 32);
    }
    tmem_wait_ld<64>(r);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster_relaxed(tmem_empty_c);

  if (EPI == EPI_BF16 || EPI == EPI_B16_OUT || EPI == EPI_T8_OUT) {
    if (c0 >= ncols) return;
    // per-tensor E4M3 operands: dequantize the accumulator with 1/(s_a s_b) of this expert
    const float alpha = Ops<EPI>::T8 ? __frcp_rn(t8_scale(a.amax_a[tl.e])) * __frcp_rn(t8_scale(a.amax_b[tl.e]))
                                     : 1.0f;
    __nv_bfloat16* orow = a.out + row * a.ldo + tl.n0 + c0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = have ? __uint_as_float(r[32 * h + i]) * alpha : 0.f;
      store_bf16x32(orow + 32 * h, v, a.out_v8);
    }
  } else if (EPI == EPI_T8_FWD_SWIGLU) {
    // per-tensor path: a = silu(g)*u*p stored as bf16 [cap][I] in out; the expert's amax of
    // the stored values is raised in amax_out (bf16 rounding is monotonic: the largest
    // stored magnitude is the rounded largest fp32 magnitude)
    const float p = a.prob_perm[row];
    const float alpha = __frcp_rn(t8_scale(a.amax_a[tl.e])) * __frcp_rn(t8_scale(a.amax_b[tl.e]));
    const int64_t col = tl.n0 + cg * 32;
    float* f = reinterpret_cast<float*>(r);
#pragma unroll
    for (int i = 0; i < 64; ++i) f[i] *= alpha;            // g | u
    if (a.gu != nullptr) {                                   // saved for the per-tensor backward
      const int64_t twoI = 2 * int64_t(a.I);
      store_bf16x32(a.gu + row * twoI + col, f, a.out_v8);
      store_bf16x32(a.gu + row * twoI + a.I + col, f + 32, a.out_v8);
    }
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      f[i] = silu_f(f[i]) * f[32 + i] * p;
      amax = max(amax, abs_bits(f[i]));
    }
    store_bf16x32(a.out + row * a.ldo + col, f, a.out_v8);
    amax = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(amax))));
    amax = __reduce_max_sync(0xFFFFFFFFu, amax);
    if (lane == 0 && amax != 0u) atomicMax(a.amax_out + tl.e, amax);
  } else if (EPI == EPI_B16_FWD_SWIGLU) {
    // bf16 path: a = silu(g)*u*p stored as bf16 [cap][I] in out (and g, u saved for the backward)
    const float p = a.prob_perm[row];
    const int64_t col = tl.n0 + cg * 32;
    float* f = reinterpret_cast<float*>(r);
    if (a.gu != nullptr) {
      const int64_t twoI = 2 * int64_t(a.I);
      store_bf16x32(a.gu + row * twoI + col, f, a.out_v8);
      store_bf16x32(a.gu + row * twoI + a.I + col, f + 32, a.out_v8);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = silu_f(f[i]) * f[32 + i] * p;
    store_bf16x32(a.out + row * a.ldo + col, f, a.out_v8);
  } else if (EPI == EPI_FWD_SWIGLU) {
    const float p = a.prob_perm[row];
    const int64_t twoI = 2 * int64_t(a.I);
    const int64_t col = tl.n0 + cg * 32;                  // column inside I
    float* f = reinterpret_cast<float*>(r);
    if (a.gu != nullptr) {
      store_bf16x32(a.gu + row * twoI + col, f, a.out_v8);
      store_bf16x32(a.gu + row * twoI + a.I + col, f + 32, a.out_v8);
    }
    const float2 p2 = make_float2(p, p);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 av = scaled_swiglu2(make_float2(f[i], f[i + 1]), make_float2(f[32 + i], f[33 + i]), p2);
      f[i] = av.x;
      f[i + 1] = av.y;
    }
    quant_row_block(f, a.q_row, a.q_row_s, row, col, a.q_row_K);
    if (a.q_col != nullptr) quant_col_block(f, a.q_col, a.q_col_s, row_blk0, col, a.cap, lane, tr);
  } else if (EPI == EPI_BWD_SWIGLU) {
    // MXFP8 SwiGLU backward: this warp's 64 columns of dA, as two halves of 32, each in two
    // passes over four chunks of eight columns.  Pass A computes dg and du (packed pairs),
    // runs the along-token quantizer rounds of the chunk (their blocks run over the warp's
    // 32 rows, so a chunk's eight columns are complete), raises the row-block maxima and
    // sums dp.  Pass B recomputes the same dg and du (the same instructions on the same
    // inputs: bit-identical) and writes their row-wise codes with the scales pass A found.
    // A chunk's dA comes from registers (columns 0..15) or from the TMEM stash, loaded one
    // chunk ahead; only one chunk is processed at a time, which keeps the epilogue within
    // its registers.  Pass B refills each chunk's g,u slot with the next half's as it frees it.
    float2 dp2 = make_float2(0.f, 0.f);
    if (have) {
      const float p = a.prob_perm[row];
      const float2 p2 = make_float2(p, p);
      const int64_t twoI = 2 * int64_t(a.I);
      const uint32_t stash = tmem_row + TM_DA_STASH + uint32_t(cg) * TM_DA_STASH_W;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int64_t col = tl.n0 + c0 + 32 * h;
        cp_async_wait_all();                               // this half's g,u are in gu_s
        float amax_g = 0.f, amax_u = 0.f;
        ColDst dst_g = col_dst(a.q_col, a.q_col_s, row_blk0, col, a.cap, lane);
        ColDst dst_u = col_dst(a.q_col, a.q_col_s, row_blk0, a.I + col, a.cap, lane);
        uint32_t dn[8];                                    // the next chunk's dA, loaded ahead
        da_issue(r, stash, h, 0, dn);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          da_land(h, j, dn);
          uint32_t d[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) d[i] = dn[i];
          if (j < 3) da_issue(r, stash, h, j + 1, dn);     // in flight during this chunk's work
          float vg[8], vu[8];
          swiglu_bwd_chunk(d, gu_s, j, lane, p2, vg, vu, &dp2);
#pragma unroll
          for (int t = 0; t < 8; t += 2) {
            amax_g = amax_raise(amax_g, vg[t], vg[t + 1]);
            amax_u = amax_raise(amax_u, vu[t], vu[t + 1]);
          }
          quant_col_round(vg, dst_g, lane, tr);
          quant_col_round(vu, dst_u, lane, tr);
          next_round(dst_g, a.cap);
          next_round(dst_u, a.cap);
        }
        const uint32_t c_g = mx_scale_code(__float_as_uint(amax_g));
        const uint32_t c_u = mx_scale_code(__float_as_uint(amax_u));
        uint8_t* row_g = a.q_row + row * twoI + col;
        uint8_t* row_u = row_g + a.I;
        uint32_t qg[8], qu[8];
        da_issue(r, stash, h, 0, dn);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          da_land(h, j, dn);
          uint32_t d[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) d[i] = dn[i];
          if (j < 3) da_issue(r, stash, h, j + 1, dn);
          float vg[8], vu[8];
          swiglu_bwd_chunk(d, gu_s, j, lane, p2, vg, vu, nullptr);
          if (h == 0) stage_gu_chunk(a, row, col + 32, gu_s, lane & 7, j);   // the next half's chunk j
          const uint2 eg = mx_encode8(vg, c_g), eu = mx_encode8(vu, c_u);
          qg[2 * j] = eg.x;
          qg[2 * j + 1] = eg.y;
          qu[2 * j] = eu.x;
          qu[2 * j + 1] = eu.y;
        }
        st_global_v8(row_g, qg);
        st_global_v8(row_u, qu);
        a.q_row_s[sf_offset(row, col >> 5, twoI)] = uint8_t(c_g);
        a.q_row_s[sf_offset(row, (a.I + col) >> 5, twoI)] = uint8_t(c_u);
      }
    }
    a.dp_part[(int64_t(tl.nb) * 4 + cg) * a.cap + row] = dp2.x + dp2.y;
  } else {  // SwiGLU backward with bf16 dH (bf16 and per-tensor operands): 64 columns as two halves of 32
    float dp = 0.f;
    if (have) {
      const float p = a.prob_perm[row];
      const int64_t twoI = 2 * int64_t(a.I);
      // per-tensor operands: dA = accumulator / (s_dY s_W)
      const float alpha =
          Ops<EPI>::T8 ? __frcp_rn(t8_scale(a.amax_a[tl.e])) * __frcp_rn(t8_scale(a.amax_b[tl.e])) : 1.0f;
      uint32_t amax = 0;
      for (int h = 0; h < 2; ++h) {
        if (h == 1) {
          tmem_ld32_async(tmem_row + TM_STASH + cg * 32, r);
          tmem_wait_ld<32>(r);
        }
        const int64_t col = tl.n0 + c0 + 32 * h;
        float o[32];
        cp_async_wait_all();                               // this half's g,u are in gu_s
        // dg = dA*p*u*silu'(g) and the row sum dp += dA*silu(g)*u
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 gw = *reinterpret_cast<const uint4*>(gu_s + ((j ^ (lane & 7)) << 4));
          const uint4 uw = *reinterpret_cast<const uint4*>(gu_s + (((4 + j) ^ (lane & 7)) << 4));
          const uint32_t gs[4] = {gw.x, gw.y, gw.z, gw.w};
          const uint32_t us[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int i = 8 * j + t;
            const float g = (t & 1) ? bf16_hi(gs[t >> 1]) : bf16_lo(gs[t >> 1]);
            const float u = (t & 1) ? bf16_hi(us[t >> 1]) : bf16_lo(us[t >> 1]);
            const float d = __uint_as_float(r[i]) * alpha;
            // the IEEE divide here: with the fast one this fully unrolled loop spills more
            const float sgm = 1.0f / (1.0f + __expf(-g));
            const float sg = g * sgm;
            dp += d * sg * u;
            o[i] = d * p * u * (sgm * (1.0f + g * (1.0f - sgm)));
            r[i] = __float_as_uint(d * p * sg);            // du = dA*p*silu(g)
          }
        }
        const float* du = reinterpret_cast<const float*>(r);
        if (h == 0) stage_gu(a, row, col + 32, gu_s, lane & 7);   // the second half, while this one is stored
        if (EPI == EPI_B16_BWD_SWIGLU) {
          store_bf16x32(a.out + row * twoI + col, o, a.out_v8);
          store_col_bf16(o, a.out_t, row_blk0, col, a.cap, lane, tr);
          store_bf16x32(a.out + row * twoI + a.I + col, du, a.out_v8);
          store_col_bf16(du, a.out_t, row_blk0, a.I + col, a.cap, lane, tr);
        } else {
          // per-tensor operands: bf16 dH rows; its codes (both orientations) come after the amax
          store_bf16x32(a.out + row * twoI + col, o, a.out_v8);
          store_bf16x32(a.out + row * twoI + a.I + col, du, a.out_v8);
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = max(amax, max(abs_bits(o[i]), abs_bits(du[i])));
        }
      }
      if (EPI == EPI_T8_BWD_SWIGLU) {
        // amax of the stored bf16 dH (bf16 rounding is monotonic), one atomic per warp
        amax = __float_as_uint(__bfloat162float(__float2bfloat16_rn(__uint_as_float(amax))));
        amax = __reduce_max_sync(0xFFFFFFFFu, amax);
        if (lane == 0 && amax != 0u) atomicMax(a.amax_out + tl.e, amax);
      }
    }
    a.dp_part[(int64_t(tl.nb) * 4 + cg) * a.cap + row] = dp;
  }
}

// B operand maps: one stacked tensor (tmB), or with PE one map per expert (each expert's
// own weight tensor; the tile decode then gives B rows inside the expert's matrix, since
// b_rows_per_expert is 0).
template <int N>
struct BMaps {
  CUtensorMap m[N];
};
constexpr int kMaxMapExperts = 128;

template <int EPI, bool PE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const __grid_constant__ BMaps<PE ? kMaxMapExperts : 1> bmaps, const GemmArgs args) {
  using L = Lay<EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + L::NSTG;
  uint64_t* tmem_full = empty + L::NSTG;         // one per accumulator buffer
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  int* seg = reinterpret_cast<int*>(smem + L::OFF_SEG);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();       // 0: leader (issues the MMAs), 1: peer
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NSTG; ++s) {
      mbar_init(&full[s], 1);                    // the leader expects both CTAs' bytes
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 2 * NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (!Ops<EPI>::NOSF) {
      prefetch_tmap(&tmSFA);
      prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_s, TMEM_COLS);          // collectively with the peer CTA
    tmem_relinquish();
  }
  // Everything above touches only this CTA's shared memory, TMEM and the parameters, so it
  // overlaps the end of the previous kernel (programmatic stream serialization); from here
  // on the kernel reads what earlier kernels wrote.  The next kernel is let in once every
  // CTA's producer has issued its last copy (or the CTA has exited): its CTAs then arrive
  // during this kernel's last tiles.
  pdl_wait();
  if (threadIdx.x == 0) {
    int acc = 0, acc_pb = 0;
    for (int e = 0; e < args.E; ++e) {
      seg[e] = acc;
      seg[SEG_PB + e] = acc_pb;
      const int rows_e = args.split_sizes != nullptr ? args.split_sizes[e] : int(args.rows_limit);
      const int nblk = (rows_e + 127) >> 7;
      acc += nblk;
      acc_pb += (nblk + 1) >> 1;
    }
    seg[args.E] = acc;
    seg[SEG_PB + args.E] = acc_pb;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                // the pair's barriers are initialised before any remote arrival
  tc_fence_after();
  if (args.mode == 1) {
    // rank of expert e: experts with more 128-token blocks, or as many and a lower id, come first
    int* order = seg + SEG_INTS;
    for (int e = threadIdx.x; e < args.E; e += blockDim.x) {
      const int me = seg[e + 1] - seg[e];
      int rank_e = 0;
      for (int f = 0; f < args.E; ++f) {
        const int other = seg[f + 1] - seg[f];
        rank_e += (other > me) || (other == me && f < e);
      }
      order[rank_e] = e;
    }
    __syncthreads();
  }
  const uint32_t tmem = *tmem_base_s;
  const int total = tile_count(args, seg);
  const uint64_t lim = args.wait_limit_ns != 0 ? args.wait_limit_ns : kWaitLimitNs;
  // the padded segments must fit the permuted capacity (rows in mode 0, K in mode 1)
  if (int64_t(seg[args.E]) * BM > args.cap) {
    if (threadIdx.x == 0) report_error(args.err, MOE_ERR_DEVICE_BOUNDS, SITE_GEMM_PRODUCER + 9);
  } else if (warp == 0) {
    if (lane == 0 && !args.selftest_no_loads) {
      // ---------------- TMA producer (both CTAs) ----------------
      const uint32_t full_c0 = mapa_shared(smem_u32(full), 0);   // the leader's full[0]
      int it = 0;
      bool issued_any = false;
      int last_round[L::NSTG];
#pragma unroll
      for (int s = 0; s < L::NSTG; ++s) last_round[s] = -1;
      bool ok = true;
      TileSrc cur, nxt;
      if (pair < total) tile_src<EPI>(args, seg, pair, rank, cur);
      for (int t = pair; t < total && ok; t += num_pairs) {
        if (t + num_pairs < total) tile_src<EPI>(args, seg, t + num_pairs, rank, nxt);
        if (PE) prefetch_tmap(&bmaps.m[cur.e]);
        for (int kt0 = 0; kt0 < cur.k_tiles; kt0 += L::PER, ++it) {
          const int st = it % L::NSTG;
          const int round = it / L::NSTG;
          if (!wait_phase(&empty[st], (round & 1) ^ 1, abort_s, args.err, SITE_GEMM_PRODUCER, lim)) {
            ok = false;
            break;
          }
          const uint32_t bar_c = full_c0 + uint32_t(st) * 8u;
          // The leader expects both CTAs' bytes; the peer's copies complete on the same barrier.
          // Every box carries the stage's full K: a short last stage (an odd number of K steps)
          // loads one K step of operands and one scale atom per box that its MMAs do not read.
          const uint32_t bytes = uint32_t(L::PER) * (A_TILE + B_HALF) + (Ops<EPI>::NOSF ? 0u : 3u * L::PER * SF_ATOM);
          if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * bytes);
          last_round[st] = round;
          issued_any = true;
          const int slot = st * L::PER;
          const int ka = cur.k0 / Ops<EPI>::KSTEP + kt0;        // first K atom of the stage
          tma_load_3d(smem + L::OFF_A + slot * A_TILE, &tmA, 0, cur.a_row, ka, bar_c);
          tma_load_3d(smem + L::OFF_B + slot * B_HALF, PE ? &bmaps.m[cur.e] : &tmB, 0, cur.b_row, ka, bar_c);
          if (!Ops<EPI>::NOSF) {
            tma_load_2d(smem + L::OFF_SFA + slot * SF_ATOM, &tmSFA, 0, cur.sfa_y + 2 * kt0, bar_c);
            tma_load_2d(smem + L::OFF_SFB0 + slot * SF_ATOM, &tmSFB, 0, cur.sfb0_y + 2 * kt0, bar_c);
            tma_load_2d(smem + L::OFF_SFB1 + slot * SF_ATOM, &tmSFB, 0, cur.sfb1_y + 2 * kt0, bar_c);
          }
        }
        cur = nxt;
      }
      pdl_launch_dependents();
      if (!ok && issued_any) {
        // let copies already issued land before the CTA exits: the leader watches the full
        // barriers (which also count the peer's copies); the peer, whose copies signal the
        // leader, gives them a fixed grace period
        if (rank == 0) {
          for (int s = 0; s < L::NSTG; ++s) {
            if (last_round[s] < 0) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&full[s], last_round[s] & 1) && globaltimer_ns() - t0 < 20000000ull) {
            }
          }
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 2000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader) ----------------
      int it = 0, tcount = 0;
      bool ok = true, issued = false;
      for (int t = pair; t < total && ok; t += num_pairs, ++tcount) {
        Tile tl;
        decode_tile<EPI>(args, seg, t, 0, tl);
        // accumulator buffer of this tile and how often it was used before
        const int ab = Ops<EPI>::ACC_BUFS == 2 ? (tcount & 1) : 0;
        const int use = Ops<EPI>::ACC_BUFS == 2 ? (tcount >> 1) : tcount;
        const uint32_t acc = tmem + TM_ACC + uint32_t(ab) * 256u;
        if (!wait_phase(&tmem_empty[ab], (use & 1) ^ 1, abort_s, args.err, SITE_GEMM_MMA_ACC, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt0 = 0; kt0 < tl.k_tiles; kt0 += L::PER, ++it) {
          const int st = it % L::NSTG;
          const int round = it / L::NSTG;
          const int nk = min(L::PER, tl.k_tiles - kt0);
          // both CTAs' operands (and scale atoms) of the stage have landed
          if (!wait_phase(&full[st], round & 1, abort_s, args.err, SITE_GEMM_MMA, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int sub = 0; sub < nk; ++sub) {
            const int slot = st * L::PER + sub;
            const int kt = kt0 + sub;
            const uint32_t tm_sfa = tmem + TM_SF0 + uint32_t(slot) * TM_SF_STRIDE;
            const uint32_t tm_sfb = tm_sfa + 4;
            if (!Ops<EPI>::NOSF) {
              // issued by this thread ahead of the MMAs that read them: executed in order
              tc_cp_sf(tm_sfa, desc_sf(smem_u32(smem + L::OFF_SFA + slot * SF_ATOM)));
              tc_cp_sf(tm_sfb, desc_sf(smem_u32(smem + L::OFF_SFB0 + slot * SF_ATOM)));
              tc_cp_sf(tm_sfb + 4, desc_sf(smem_u32(smem + L::OFF_SFB1 + slot * SF_ATOM)));
            }
            const uint64_t adesc = desc_sw128(smem_u32(smem + L::OFF_A + slot * A_TILE));
            const uint64_t bdesc = desc_sw128(smem_u32(smem + L::OFF_B + slot * B_HALF));
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk) {
              // +32 bytes along K inside the 128-byte swizzle atom = +2 in the encoded start address
              if (Ops<EPI>::B16) {
                tc_mma_bf16(acc, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc_bf16(BN),
                            (kt | kk) != 0);
                continue;
              }
              if (Ops<EPI>::T8) {
                tc_mma_f8(acc, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc_f8(BN), (kt | kk) != 0);
                continue;
              }
              tc_mma_mxf8(acc, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc_mxf8(BN, kk), tm_sfa,
                          tm_sfb, (kt | kk) != 0);
            }
          }
          issued = true;
          tc_commit(&empty[st]);                 // frees the stage in both CTAs
        }
        if (!ok) break;
        tc_commit(&tmem_full[ab]);               // both halves of the accumulator are ready
      }
      if (!ok && issued) {
        tc_commit(drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 20000000ull) {
        }
      }
    }
  } else {
    // ---------------- epilogue warps 2..17 (both CTAs) ----------------
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int cg = (warp - 2) >> 2;            // column group 0..3
    const uint32_t tmem_row = tmem + (uint32_t(q * 32) << 16);
    const uint32_t tmem_empty_c0 = mapa_shared(smem_u32(tmem_empty), 0);
    float* tr = reinterpret_cast<float*>(smem + L::OFF_TR) + (warp - 2) * TR_WARP_FLOATS;
    uint8_t* gu_s = smem + L::OFF_GU + (warp - 2) * L::GU_WARP + lane * GU_PITCH;
    int tcount = 0;
    for (int t = pair; t < total; t += num_pairs, ++tcount) {
      Tile tl;
      decode_tile<EPI>(args, seg, t, int(rank), tl);
      if (Ops<EPI>::SWIGLU_BWD && tl.valid && cg * 64 < (tl.second ? 256 : 128)) {
        // this lane's saved g and u of the first half land in shared memory while the MMAs run
        stage_gu(args, tl.out_row + q * 32 + lane, tl.n0 + cg * 64, gu_s, lane & 7);
      }
      const int ab = Ops<EPI>::ACC_BUFS == 2 ? (tcount & 1) : 0;
      const int use = Ops<EPI>::ACC_BUFS == 2 ? (tcount >> 1) : tcount;
      if (!wait_phase(&tmem_full[ab], use & 1, abort_s, args.err, SITE_GEMM_EPILOGUE, lim)) break;
      tc_fence_after();
      epilogue_tile<EPI>(args, tl, tmem_row + uint32_t(ab) * 256u, q, cg, lane, tmem_empty_c0 + uint32_t(ab) * 8u,
                         tr, gu_s);
    }
    if (Ops<EPI>::SWIGLU_BWD) cp_async_wait_all();   // nothing in flight when a wait gave up
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                // no CTA leaves while the pair's MMAs or arrivals may touch it
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---- self-tests of the epilogue's parts ----------------------------------------------
// The epilogue quantizers on caller data: warp w of a CTA takes the 32-row x 32-column
// block (bx*4 + w) of an f32 [rows][cols] tensor, each lane one row's 32 values, exactly
// as an epilogue warp holds them, and calls the epilogue's row-wise and along-token
// quantizers on them.
constexpr int EQ_WARPS = 4;
__global__ void __launch_bounds__(32 * EQ_WARPS) epilogue_quant_selftest_kernel(
    const float* __restrict__ src, int rows, int cols, uint8_t* codes, uint8_t* scales, uint8_t* codes_t,
    uint8_t* scales_t) {
  __shared__ float tr_all[EQ_WARPS * TR_WARP_FLOATS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t blk = int64_t(blockIdx.x) * EQ_WARPS + warp;
  const int cb = cols / 32;
  if (blk >= int64_t(rows / 32) * cb) return;                  // warp-uniform
  const int64_t row_blk0 = (blk / cb) * 32;
  const int64_t col = (blk % cb) * 32;
  const int64_t row = row_blk0 + lane;
  float v[32];
  const float4* p = reinterpret_cast<const float4*>(src + row * cols + col);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = p[i];
    v[4 * i + 0] = q.x;
    v[4 * i + 1] = q.y;
    v[4 * i + 2] = q.z;
    v[4 * i + 3] = q.w;
  }
  quant_row_block(v, codes, scales, row, col, cols);
  quant_col_block(v, codes_t, scales_t, row_blk0, col, rows, lane, tr_all + warp * TR_WARP_FLOATS);
}

// The MXFP8 tensor pipe's issue ceiling: CTA pairs (one CTA per SM) issue the GEMM's
// MMAs -- per 128-deep K step three scale-factor copies and four
// tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale of M=256, N=256, K=32 --
// back to back on operands that stay in shared memory (zeros), with no loads and no
// epilogue.  FLOPs per K step and pair: 2 * 256 * 256 * 128.
constexpr int MR_THREADS = 64;
constexpr int MR_OFF_A = 0, MR_OFF_B = A_TILE, MR_OFF_SF = A_TILE + B_HALF;
constexpr int MR_OFF_BAR = MR_OFF_SF + 3 * SF_ATOM;
constexpr int MR_SMEM_USED = MR_OFF_BAR + 64 + 1024;
// requested so that a second CTA never fits on an SM: one CTA (and one TMEM allocation) per SM
constexpr int MR_SMEM = 160 * 1024;
static_assert(MR_SMEM_USED <= MR_SMEM, "self-test shared memory");
__global__ void __launch_bounds__(MR_THREADS, 1) mma_rate_selftest_kernel(int k_steps, int* err, uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + MR_OFF_BAR);
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + MR_OFF_BAR + 8);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + MR_OFF_BAR + 12);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  for (int i = threadIdx.x; i < MR_OFF_BAR / 16; i += MR_THREADS) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the zeros are visible to the tensor pipe
  if (warp == 1) {
    tmem_alloc(tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  if (warp == 0 && lane == 0 && rank == 0) {
    const uint32_t tm_sfa = tmem + TM_SF0, tm_sfb = tm_sfa + 4;
    const uint64_t adesc = desc_sw128(smem_u32(smem + MR_OFF_A));
    const uint64_t bdesc = desc_sw128(smem_u32(smem + MR_OFF_B));
    for (int kt = 0; kt < k_steps; ++kt) {
      tc_cp_sf(tm_sfa, desc_sf(smem_u32(smem + MR_OFF_SF)));
      tc_cp_sf(tm_sfb, desc_sf(smem_u32(smem + MR_OFF_SF + SF_ATOM)));
      tc_cp_sf(tm_sfb + 4, desc_sf(smem_u32(smem + MR_OFF_SF + 2 * SF_ATOM)));
#pragma unroll
      for (int kk = 0; kk < BK / 32; ++kk)
        tc_mma_mxf8(tmem + TM_ACC, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc_mxf8(BN, kk), tm_sfa,
                    tm_sfb, (kt | kk) != 0);
    }
    tc_commit(done);                               // arrives in both CTAs once every MMA is done
  }
  if (threadIdx.x == 0) wait_phase(done, 0, abort_s, err, SITE_GEMM_DRAIN + 5, limit_ns);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---- router weight gradient on the tensor cores --------------------------------------
// dW_r^T[h][e] = sum_t x[t][h] * dl[t][e] (the router's weight gradient, transposed) for
// one 128-row block of h and one chunk of tokens per CTA, single-CTA MMAs
// (cta_group::1, M = 128, N = roundup(E, 64)).  x [T][H] and dl [T][N] both keep the
// MMA's M / N index contiguous, so TMA loads them as they lie into MN-major 128-byte
// swizzled tiles: 64 tokens (K) x 64 columns per box, boxes of further 64-column blocks
// LBO apart, 8-token groups 1024 bytes apart (SBO).  dl arrives as two bf16 terms hi + lo
// (hi = bf16(dl), lo = bf16(dl - hi): dl to about 2^-17 relative); each 16-token step
// issues hi . x and lo . x into the same f32 accumulator.  Chunk c's tile is written to
// partial[c][e][h]; the chunks are summed in chunk order by a separate reduction.
constexpr int RDW_KT = 64;                     // tokens per pipeline stage
constexpr int RDW_M = 128;                     // hidden rows of a tile
constexpr int RDW_MAX_STG = 8;
constexpr uint32_t RDW_SMEM_MAX = 200u * 1024u;
constexpr uint32_t RDW_A_BYTES = RDW_M * RDW_KT * 2;   // two 64-column boxes of x

struct RouterDwArgs {
  int H, E, N;            // N = roundup(E, 64): accumulator columns
  int nst, per;           // 64-token stages in all, and per chunk
  int stages;             // pipeline depth
  float* partial;         // [chunks][E][H]
  int* err;
};

__device__ __forceinline__ void tma_load_2d_cta(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_cta(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_cta() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_cta(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit_cta(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_cta(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// MN-major operand with 128-byte swizzle: rows of 128 bytes (64 bf16 of the M or N index)
// per K index, 8-row groups every 1024 bytes (SBO), 64-column blocks every lbo bytes.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}
// kind::f16 instruction descriptor: bf16 x bf16 -> f32, A and B MN-major (transposed).
__device__ __forceinline__ uint32_t idesc_bf16_mn(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

__global__ void __launch_bounds__(192, 1) router_dw_tc_kernel(const __grid_constant__ CUtensorMap mx,
                                                              const __grid_constant__ CUtensorMap mhi,
                                                              const __grid_constant__ CUtensorMap mlo,
                                                              const RouterDwArgs a) {
  extern __shared__ uint8_t rdw_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rdw_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[RDW_MAX_STG], empty[RDW_MAX_STG], done;
  __shared__ uint32_t tmem_s;
  __shared__ int abort_flag;
  volatile int* abort_s = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NB = a.N / 64;
  const uint32_t b_bytes = uint32_t(a.N) * RDW_KT * 2;
  const uint32_t stage_bytes = RDW_A_BYTES + 2 * b_bytes;
  const uint32_t ncols = a.N <= 64 ? 64u : a.N <= 128 ? 128u : 256u;
  const int h0 = blockIdx.x * RDW_M, c = blockIdx.y;
  const int s0 = c * a.per;
  const int n = min(a.nst, s0 + a.per) - s0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc_cta(&tmem_s, ncols);
    tmem_relinquish_cta();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      prefetch_tmap(&mx);
      prefetch_tmap(&mhi);
      prefetch_tmap(&mlo);
      int last_round[RDW_MAX_STG];
#pragma unroll
      for (int s = 0; s < RDW_MAX_STG; ++s) last_round[s] = -1;
      bool ok = true;
      for (int i = 0; i < n; ++i) {
        const int slot = i % a.stages, round = i / a.stages;
        if (!wait_phase(&empty[slot], (round & 1) ^ 1, abort_s, a.err, SITE_ROUTER_DW, kWaitLimitNs)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + size_t(slot) * stage_bytes;
        mbar_arrive_expect_tx(&full[slot], stage_bytes);
        const int t = (s0 + i) * RDW_KT;
        tma_load_2d_cta(st, &mx, h0, t, &full[slot]);
        tma_load_2d_cta(st + 8192, &mx, h0 + 64, t, &full[slot]);
        for (int j = 0; j < NB; ++j) {
          tma_load_2d_cta(st + RDW_A_BYTES + j * 8192, &mhi, 64 * j, t, &full[slot]);
          tma_load_2d_cta(st + RDW_A_BYTES + b_bytes + j * 8192, &mlo, 64 * j, t, &full[slot]);
        }
        last_round[slot] = round;
      }
      if (!ok) {
        // copies already issued land before the CTA exits (bounded)
        for (int s = 0; s < a.stages; ++s) {
          if (last_round[s] < 0) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[s], last_round[s] & 1) && globaltimer_ns() - t0 < 20000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = idesc_bf16_mn(RDW_M, a.N);
      for (int i = 0; i < n; ++i) {
        const int slot = i % a.stages, round = i / a.stages;
        if (!wait_phase(&full[slot], round & 1, abort_s, a.err, SITE_ROUTER_DW + 1, kWaitLimitNs)) break;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + size_t(slot) * stage_bytes);
        const uint64_t ad = desc_sw128_mn(st, 8192);
        const uint64_t bh = desc_sw128_mn(st + RDW_A_BYTES, 8192);
        const uint64_t bl = desc_sw128_mn(st + RDW_A_BYTES + b_bytes, 8192);
#pragma unroll
        for (int kk = 0; kk < RDW_KT / 16; ++kk) {
          // 16 tokens = two 8-row groups = 2048 bytes, 128 in the descriptor's 16-byte units
          tc_mma_bf16_cta(tmem, ad + uint64_t(128 * kk), bh + uint64_t(128 * kk), idesc, (i | kk) != 0);
          tc_mma_bf16_cta(tmem, ad + uint64_t(128 * kk), bl + uint64_t(128 * kk), idesc, 1);
        }
        tc_commit_cta(&empty[slot]);
      }
      tc_commit_cta(&done);                    // arrives once every MMA issued above is complete
    }
  } else {
    // ---------------- epilogue warps 2..5: warp w reads TMEM lanes 32*(w%4).. ----------------
    const int q = warp & 3;
    const int h = h0 + 32 * q + lane;
    bool ok = wait_phase(&done, 0, abort_s, a.err, SITE_ROUTER_DW + 2, kWaitLimitNs);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok) {
      tc_fence_after();
      for (int j0 = 0; j0 < a.N; j0 += 16) {
        uint32_t r[16];
        tmem_ld16_async(tmem + (uint32_t(32 * q) << 16) + uint32_t(j0), r);
        tmem_wait_ld<16>(r);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int e = j0 + jj;
          if (e < a.E && h < a.H) a.partial[(int64_t(c) * a.E + e) * a.H + h] = __uint_as_float(r[jj]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_s) {
    // an MMA may still run after a wait gave up: let it finish before the memory goes (bounded)
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&done, 0) && globaltimer_ns() - t0 < 20000000ull) {
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_cta(tmem, ncols);
}

// ---- router logits on the tensor cores ---------------------------------------------------
// logits[t][e] = sum_h x[t][h] * W_r[e][h] for 128 tokens per CTA: single-CTA MMAs (M = 128,
// N = roundup(E, 16) experts, f32 accumulation in TMEM), both operands K-major by TMA (x
// [T][H] and W_r [E][H] as they lie, 64 bf16 of K per 128-byte swizzled row).  The W_r box
// holds E rows; rows E..N-1 of the staged tile are stale and feed only output columns past
// E, which are never written.  Bound by reading x once.
constexpr int RF_KT = 64;                      // K elements (bf16) per stage
constexpr int RF_M = 128;                      // tokens per CTA
constexpr int RF_MAX_STG = 8;

struct RouterFwdArgs {
  int T, E, N;            // N = roundup(E, 16): accumulator columns
  int nk;                 // 64-wide K chunks (H / 64)
  int steps;              // K chunks per pipeline stage (more bytes behind each barrier)
  int stages;             // pipeline depth
  float* logits;          // [T][E]
  int* err;
};

__device__ __forceinline__ uint32_t idesc_bf16_m128(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(RF_M >> 4) << 24);
}

__global__ void __launch_bounds__(192, 1) router_fwd_tc_kernel(const __grid_constant__ CUtensorMap mx,
                                                               const __grid_constant__ CUtensorMap mw,
                                                               const RouterFwdArgs a) {
  extern __shared__ uint8_t rf_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rf_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[RF_MAX_STG], empty[RF_MAX_STG], done;
  __shared__ uint32_t tmem_s;
  __shared__ int abort_flag;
  volatile int* abort_s = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t A_BYTES = RF_M * RF_KT * 2;                     // 16 KB
  const uint32_t b_slot = (uint32_t(a.N) * RF_KT * 2 + 1023u) & ~1023u;   // the N-row tile of a chunk
  const uint32_t b_bytes = uint32_t(a.E) * RF_KT * 2;                     // what the E-row box brings
  const uint32_t chunk_bytes = A_BYTES + b_slot;
  const uint32_t stage_bytes = uint32_t(a.steps) * chunk_bytes;
  const int n_st = (a.nk + a.steps - 1) / a.steps;                          // pipeline stages of the CTA
  const uint32_t ncols = a.N <= 32 ? 32u : a.N <= 64 ? 64u : a.N <= 128 ? 128u : 256u;
  const int t0 = blockIdx.x * RF_M;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc_cta(&tmem_s, ncols);
    tmem_relinquish_cta();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      prefetch_tmap(&mx);
      prefetch_tmap(&mw);
      int last_round[RF_MAX_STG];
#pragma unroll
      for (int s = 0; s < RF_MAX_STG; ++s) last_round[s] = -1;
      bool ok = true;
      for (int i = 0; i < n_st; ++i) {
        const int slot = i % a.stages, round = i / a.stages;
        if (!wait_phase(&empty[slot], (round & 1) ^ 1, abort_s, a.err, SITE_ROUTER_DW + 10, kWaitLimitNs)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + size_t(slot) * stage_bytes;
        const int c0 = i * a.steps, nc = min(a.steps, a.nk - c0);
        mbar_arrive_expect_tx(&full[slot], uint32_t(nc) * (A_BYTES + b_bytes));
        for (int c = 0; c < nc; ++c) {
          tma_load_2d_cta(st + c * chunk_bytes, &mx, (c0 + c) * RF_KT, t0, &full[slot]);
          tma_load_2d_cta(st + c * chunk_bytes + A_BYTES, &mw, (c0 + c) * RF_KT, 0, &full[slot]);
        }
        last_round[slot] = round;
      }
      if (!ok) {
        for (int s = 0; s < a.stages; ++s) {
          if (last_round[s] < 0) continue;
          const uint64_t tw = globaltimer_ns();
          while (!mbar_try_wait(&full[s], last_round[s] & 1) && globaltimer_ns() - tw < 20000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = idesc_bf16_m128(a.N);
      for (int i = 0; i < n_st; ++i) {
        const int slot = i % a.stages, round = i / a.stages;
        if (!wait_phase(&full[slot], round & 1, abort_s, a.err, SITE_ROUTER_DW + 11, kWaitLimitNs)) break;
        tc_fence_after();
        const int c0 = i * a.steps, nc = min(a.steps, a.nk - c0);
        for (int c = 0; c < nc; ++c) {
          const uint32_t st = smem_u32(smem + size_t(slot) * stage_bytes + size_t(c) * chunk_bytes);
          const uint64_t ad = desc_sw128(st);
          const uint64_t bd = desc_sw128(st + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < RF_KT / 16; ++kk)
            // 16 bf16 of K = 32 bytes inside the 128-byte swizzle row = +2 in the encoded address
            tc_mma_bf16_cta(tmem, ad + uint64_t(2 * kk), bd + uint64_t(2 * kk), idesc, (i | c | kk) != 0);
        }
        tc_commit_cta(&empty[slot]);
      }
      tc_commit_cta(&done);
    }
  } else {
    // ---------------- epilogue warps 2..5: warp w reads TMEM lanes 32*(w%4).. (tokens) ----------------
    const int q = warp & 3;
    const int t = t0 + 32 * q + lane;
    bool ok = wait_phase(&done, 0, abort_s, a.err, SITE_ROUTER_DW + 12, kWaitLimitNs);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok) {
      tc_fence_after();
      float* orow = a.logits + int64_t(t) * a.E;
      for (int j0 = 0; j0 < a.N; j0 += 16) {
        uint32_t r[16];
        tmem_ld16_async(tmem + (uint32_t(32 * q) << 16) + uint32_t(j0), r);
        tmem_wait_ld<16>(r);
        if (t < a.T) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (j0 + jj < a.E) orow[j0 + jj] = __uint_as_float(r[jj]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_s) {
    const uint64_t tw = globaltimer_ns();
    while (!mbar_try_wait(&done, 0) && globaltimer_ns() - tw < 20000000ull) {
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_cta(tmem, ncols);
}

// ---- host side -----------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D map over a row-major [rows][K] tensor: {128 bytes of K, rows, K / 128-byte atoms}
// with strides {row pitch, 128 bytes}; box {128 bytes, 128 rows, STAGE_STEPS atoms}.
// One copy fetches a barrier stage's K steps of 128 rows: TMA delivery per SM grows
// with the bytes per copy as well as per barrier stage.
bool encode_map3(CUtensorMap* m, const void* base, int64_t rows, int64_t K, bool b16) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  const int64_t esize = b16 ? 2 : 1;
  cuuint64_t dims[3] = {cuuint64_t(BK / esize), cuuint64_t(rows), cuuint64_t(K * esize / BK)};
  cuuint64_t strides[2] = {cuuint64_t(K * esize), cuuint64_t(BK)};
  cuuint32_t box[3] = {cuuint32_t(BK / esize), 128, cuuint32_t(STAGE_STEPS)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, b16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over n_atoms 512-byte scale atoms seen as [2 * n_atoms][256] bytes: one
// {256, 2 * STAGE_STEPS} box is the consecutive atoms of a barrier stage's K steps
// (row 2i = atom i); no swizzle, so the atoms land in shared memory byte for byte.
bool encode_sf_map(CUtensorMap* m, const void* base, int64_t n_atoms) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {256, cuuint64_t(2 * n_atoms)};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 2 * STAGE_STEPS};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, bool PE>
cudaError_t launch_epi(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msfa,
                       const CUtensorMap& msfb, const BMaps<PE ? kMaxMapExperts : 1>& bmaps, const GemmArgs& a,
                       int grid, cudaStream_t st) {
  // the shared-memory attribute is per device: set it once on each device this process uses
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, PE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<EPI>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_release);
  }
  // CTA pairs: clusters of two along x
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Lay<EPI>::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // the kernel calls pdl_wait()
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<EPI, PE>, ma, mb, msfa, msfb, bmaps, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_kind(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msfa,
                        const CUtensorMap& msfb, const BMaps<kMaxMapExperts>* pe_maps, const GemmArgs& a, int grid,
                        cudaStream_t st) {
  // one B map per expert: the bf16 forward kinds (they read the master weights as they are)
  if constexpr (EPI == EPI_B16_OUT || EPI == EPI_B16_FWD_SWIGLU) {
    if (pe_maps != nullptr) return launch_epi<EPI, true>(ma, mb, msfa, msfb, *pe_maps, a, grid, st);
  }
  if (pe_maps != nullptr) return cudaErrorInvalidValue;
  const BMaps<1> none{mb};
  return launch_epi<EPI, false>(ma, mb, msfa, msfb, none, a, grid, st);
}

}  // namespace

// 2-D map over a row-major bf16 [rows][cols] tensor for four-row gathers: box one row
// high and box_cols wide, no swizzle (the rows land back to back in shared memory).
// A row coordinate >= rows reads zeros.
bool encode_gather_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {cuuint32_t(box_cols), 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_epilogue_quant_selftest(const float* src, int rows, int cols, uint8_t* codes, uint8_t* scales,
                                           uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st) {
  const int64_t blocks = int64_t(rows / 32) * (cols / 32);
  const int64_t grid = (blocks + EQ_WARPS - 1) / EQ_WARPS;
  epilogue_quant_selftest_kernel<<<unsigned(grid), 32 * EQ_WARPS, 0, st>>>(src, rows, cols, codes, scales, codes_t,
                                                                           scales_t);
  return cudaGetLastError();
}

cudaError_t launch_mma_rate_selftest(int k_steps, int* err, int* pairs, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mma_rate_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MR_SMEM);
  if (e != cudaSuccess) return e;
  *pairs = sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * (sms / 2)));
  cfg.blockDim = dim3(MR_THREADS);
  cfg.dynamicSmemBytes = MR_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mma_rate_selftest_kernel, k_steps, err, kWaitLimitNs);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(int epi, const GemmArgs& args, const void* A, int64_t a_rows, int64_t a_K,
                                const void* B, int64_t b_rows, int64_t b_K, int64_t max_tiles, cudaStream_t st,
                                char* msg, size_t msg_len, const void* const* b_experts) {
  if (max_tiles <= 0) return cudaSuccess;
  GemmArgs a = args;
  const auto al32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
  a.out_v8 = al32(a.out) && al32(a.out_t) && al32(a.gu);
  // one B map per expert: b_experts[e] is expert e's [b_rows][b_K] matrix
  static thread_local BMaps<kMaxMapExperts> pe_maps;
  if (b_experts != nullptr) {
    if (a.E > kMaxMapExperts || a.b_rows_per_expert != 0) {
      snprintf(msg, msg_len, "per-expert weight tensors: E=%d must be <= %d", a.E, kMaxMapExperts);
      return cudaErrorInvalidValue;
    }
    const bool b16e = (epi == EPI_B16_OUT || epi == EPI_B16_FWD_SWIGLU);
    for (int e = 0; e < a.E; ++e) {
      if (!encode_map3(&pe_maps.m[e], b_experts[e], b_rows, b_K, b16e)) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed for expert %d's weight (%lld x %lld)", e,
                 (long long)b_rows, (long long)b_K);
        return cudaErrorInvalidValue;
      }
    }
    for (int e = a.E; e < kMaxMapExperts; ++e) pe_maps.m[e] = pe_maps.m[0];
  }
  CUtensorMap ma, mb, msfa, msfb;
  const bool b16 = (epi == EPI_B16_OUT || epi == EPI_B16_FWD_SWIGLU || epi == EPI_B16_BWD_SWIGLU);
  const bool t8 = (epi == EPI_T8_OUT || epi == EPI_T8_FWD_SWIGLU || epi == EPI_T8_BWD_SWIGLU);
  if (!encode_map3(&ma, A, a_rows, a_K, b16) || !encode_map3(&mb, B, b_rows, b_K, b16)) {
    snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (A %lld x %lld, B %lld x %lld)", (long long)a_rows,
             (long long)a_K, (long long)b_rows, (long long)b_K);
    return cudaErrorInvalidValue;
  }
  if (b16 || t8) {
    msfa = ma;                                   // no scale factors: never read
    msfb = ma;
  } else if (!encode_sf_map(&msfa, a.sfa, (a_rows / 128) * (a.sfa_K / BK)) ||
             !encode_sf_map(&msfb, a.sfb, (b_rows / 128) * (a.sfb_K / BK))) {
    snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed for the scale atoms (A %lld x %lld, B %lld x %lld)",
             (long long)a_rows, (long long)a.sfa_K, (long long)b_rows, (long long)a.sfb_K);
    return cudaErrorInvalidValue;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // persistent CTA pairs: at most one pair per two SMs, no more pairs than 128-row tiles
  const int64_t pairs_max = sms / 2;
  const int grid = 2 * int(max_tiles < pairs_max ? max_tiles : pairs_max);
  switch (epi) {
    case EPI_BF16: return launch_kind<EPI_BF16>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_FWD_SWIGLU: return launch_kind<EPI_FWD_SWIGLU>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_BWD_SWIGLU: return launch_kind<EPI_BWD_SWIGLU>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_B16_OUT: return launch_kind<EPI_B16_OUT>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_B16_FWD_SWIGLU: return launch_kind<EPI_B16_FWD_SWIGLU>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_T8_OUT: return launch_kind<EPI_T8_OUT>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_T8_FWD_SWIGLU: return launch_kind<EPI_T8_FWD_SWIGLU>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_B16_BWD_SWIGLU: return launch_kind<EPI_B16_BWD_SWIGLU>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    case EPI_T8_BWD_SWIGLU: return launch_kind<EPI_T8_BWD_SWIGLU>(ma, mb, msfa, msfb, b_experts != nullptr ? &pe_maps : nullptr, a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}


// ---- router weight gradient: host side -----------------------------------------------
int router_dw_cols(int E) { return (E + 63) / 64 * 64; }
int router_dw_max_chunks(int H) {
  const int tiles = (H + RDW_M - 1) / RDW_M;
  const int c = 256 / tiles;
  return c < 1 ? 1 : c > 32 ? 32 : c;
}

static bool encode_map_bf16_2d(CUtensorMap* m, const void* base, int64_t inner, int64_t outer) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  cuuint64_t strides[1] = {cuuint64_t(inner * 2)};
  cuuint32_t box[2] = {64, cuuint32_t(RDW_KT)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_router_dw_tc(const void* x, const void* dl_hi, const void* dl_lo, int T, int H, int E,
                                float* partial, int max_chunks, int* chunks_used, int* err, cudaStream_t st) {
  if (H % RDW_M != 0 || T < 1 || E < 1 || E > 256) return cudaErrorInvalidValue;
  const int N = router_dw_cols(E);
  CUtensorMap mx, mhi, mlo;
  if (!encode_map_bf16_2d(&mx, x, H, T) || !encode_map_bf16_2d(&mhi, dl_hi, N, T) ||
      !encode_map_bf16_2d(&mlo, dl_lo, N, T))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int tiles = H / RDW_M;
  const int nst = (T + RDW_KT - 1) / RDW_KT;
  int S = sms / tiles;
  S = S < 1 ? 1 : S;
  S = S > max_chunks ? max_chunks : S;
  S = S > nst ? nst : S;
  const int per = (nst + S - 1) / S;
  S = (nst + per - 1) / per;                   // every chunk holds at least one stage
  RouterDwArgs a{};
  a.H = H;
  a.E = E;
  a.N = N;
  a.nst = nst;
  a.per = per;
  a.partial = partial;
  a.err = err;
  const uint32_t stage_bytes = RDW_A_BYTES + 2u * uint32_t(N) * RDW_KT * 2u;
  int stages = int(RDW_SMEM_MAX / stage_bytes);
  a.stages = stages > RDW_MAX_STG ? RDW_MAX_STG : stages;
  const size_t smem = size_t(a.stages) * stage_bytes + 1024;
  e = cudaFuncSetAttribute(router_dw_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  router_dw_tc_kernel<<<dim3(unsigned(tiles), unsigned(S)), 192, smem, st>>>(mx, mhi, mlo, a);
  *chunks_used = S;
  return cudaGetLastError();
}


// ---- router logits: host side --------------------------------------------------------------
static bool encode_map_bf16_kmajor(CUtensorMap* m, const void* base, int64_t K, int64_t rows, int box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(K * 2)};
  cuuint32_t box[2] = {cuuint32_t(RF_KT), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_router_fwd_tc(const void* x, const void* w, int T, int H, int E, float* logits, int* err,
                                 cudaStream_t st) {
  if (T < 1 || E < 1 || E > 256 || H % RF_KT != 0) return cudaErrorInvalidValue;
  RouterFwdArgs a{};
  a.T = T;
  a.E = E;
  a.N = (E + 15) / 16 * 16;
  a.nk = H / RF_KT;
  a.logits = logits;
  a.err = err;
  CUtensorMap mx, mw;
  if (!encode_map_bf16_kmajor(&mx, x, H, T, RF_M) || !encode_map_bf16_kmajor(&mw, w, H, E, E))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e0 != cudaSuccess) return e0;
  // more CTAs than SMs: half the shared memory each, two CTAs per SM, one wave
  const int ctas = (T + RF_M - 1) / RF_M;
  const uint32_t budget = ctas > sms ? RDW_SMEM_MAX / 2 : RDW_SMEM_MAX;
  const uint32_t chunk = uint32_t(RF_M) * RF_KT * 2 + ((uint32_t(a.N) * RF_KT * 2 + 1023u) & ~1023u);
  // at least three stages, each with as many 64-wide K chunks as fit (at most four)
  int steps = int(budget / (3 * chunk));
  steps = steps < 1 ? 1 : steps > 4 ? 4 : steps;
  a.steps = steps;
  const uint32_t stage_bytes = uint32_t(steps) * chunk;
  const int stages = int(budget / stage_bytes);
  a.stages = stages > RF_MAX_STG ? RF_MAX_STG : stages;
  const size_t smem = size_t(a.stages) * stage_bytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(router_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  router_fwd_tc_kernel<<<unsigned((T + RF_M - 1) / RF_M), 192, smem, st>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace moe
