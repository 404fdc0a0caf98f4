// mla_decode.cu — split-KV flash-decoding of MLA over the paged latent cache
// (plan kernel and decode kernel; the partials are merged by mla_combine.cu).
//
// Method: MLA operator write-up (nxmr.cn/news/151634) §1 (cache row = 512-d
// latent + 64-d RoPE key), §3 (64-token pages, a tile of 64 tokens, a
// multi-stage copy pipeline) and §4 (matrix absorption: scores are
// q_abs . c_KV + q_R . k_R, so attention runs in the 576-d latent space and
// the cache is never decompressed).
//
// GB300 design of the decode kernel
//   * Query rows (l, h) form the M = 128 dimension of tcgen05 MMAs; a page
//     of 64 tokens is the N (scores) or K (values) dimension.
//   * An fp32 accumulator O of 128 rows x 512 latents would fill all 512
//     tensor-memory columns of an SM, so each 128-row block runs on a CTA
//     PAIR (cluster rank bit 0 = r): CTA r owns latent half r (256 columns of
//     O) and loads only its half of each page plus half of the 64 RoPE
//     columns.  Each CTA computes a partial score tile over its columns
//     (fp32 in tensor memory), converts it to 16-bit fixed point with a
//     power-of-two scale per query row and sends it to the peer with one
//     bulk shared-to-shared copy per TMEM lane quadrant (16 KiB + 512 B of
//     scales per page).  Each CTA adds its own fp32 partial to the peer's
//     dequantised one; the two CTAs' scores differ by at most 2^-14 of the
//     row's largest partial, and each CTA normalises its half of O by its
//     own row sums, so each half is an exact softmax average of slightly
//     different weights.  The exchange is double-buffered and the softmax
//     warps run one page behind it, so the copy of page q overlaps the
//     softmax of page q-1.
//   * Tensor memory per CTA (all 512 columns): O (256) | Q latent half (128,
//     bf16 pairs, the MMA A operand) | two score tiles S (64 each).  The
//     RoPE half of Q is a 64-byte swizzled tile in shared memory (A operand
//     of the last two K steps).  The page tile in shared memory is used
//     twice: K-major as B for S = Q.K^T and MN-major as B for O += P.V.
//   * P (bf16) is written by the softmax warps into the receive slot whose
//     peer partial they have just read, row for row, as the K-major
//     128-byte-swizzled A operand of P.V.
//   * The first segment's query arrives by TMA ahead of the first page: its
//     latent half into the four (still idle) exchange slots, whence the
//     softmax warps move it into tensor memory, and its RoPE half into its
//     shared-memory tile.  Later segments' queries are loaded by the softmax
//     warps with plain loads (RoPE tile by TMA).  The exchange slots are
//     handed to the peer (a relaxed remote arrive on its "can send"
//     barriers) only once the query has left them.
//   * Pages arrive by TMA (four 64 x 64 latent boxes with 128-byte swizzle,
//     one 32 x 64 RoPE box with 64-byte swizzle) into a 4-stage mbarrier
//     ring; one thread issues QK MMAs, one issues P.V MMAs, one issues
//     copies, four exchange warps move partial scores, eight softmax warps
//     (two per TMEM lane quadrant, one query row and half the page's keys
//     per thread) do the masking, online softmax and epilogue.  Rescaling of
//     O after a new row maximum is deferred until the maximum has grown by
//     2^8 (log2 units), so it is rare.
//   * Split-KV: the pages of all sequences, in order, are cut into equal
//     contiguous ranges, one per cluster; a range that covers parts of several
//     sequences yields one partial (o, lse) per sequence, stored in slot
//     b + unit (o chunk-major, [slot][column/4][row][4] fp32).  mla_combine.cu
//     merges them, alone or inside the W_UV projection.
//   * FP8 cache (mla_decode_paged_fp8): rows of 512 E4M3 codes, the bf16
//     RoPE key and four fp32 power-of-two scales (656 bytes).  The codes and
//     scales land in a raw slot, the RoPE columns in a ring slot; a
//     dequantising warp writes code * scale as f16 into the stage, in the
//     layout the bf16 cache's tiles have, so the latent K steps and P.V run
//     as f16 MMAs (query and P in f16), the RoPE K steps as bf16 MMAs into
//     the same fp32 scores.  HBM bytes per token: 656 against 1152.
//   * Every wait is bounded (wall clock).  A wait that gives up records
//     MLA_ERR_TIMEOUT in the workspace status word and raises the abort flag
//     of both CTAs of the pair; every role then leaves its loop, and the
//     teardown waits (ignoring the flag) for every copy and MMA this CTA
//     started and every exchange copy the peer sent it, frees tensor memory
//     and returns.
#include <climits>
#include <cmath>
#include <mutex>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

namespace {
constexpr int kStages = 4;
constexpr int kBoxBytes = kPage * 64 * 2;       // 64 tokens x 64 bf16 = 8 KiB, 128-byte swizzle
constexpr int kRopeBoxBytes = kPage * 32 * 2;   // 64 tokens x 32 bf16 = 4 KiB, 64-byte swizzle
constexpr int kXRowBytes = kPage * 2;           // one query row's 64 partial scores, int16
constexpr int kXQuadBytes = 32 * kXRowBytes;    // the 32 rows of one TMEM lane quadrant, 4 KiB
constexpr int kXSlot = 4 * kXQuadBytes;         // exchange slot: 128 rows x 64 int16 = 16 KiB
constexpr int kXScaleBytes = 32 * 4;            // a quadrant's 32 row scales (fp32), 128 B
constexpr int kXQuadTx = kXQuadBytes + kXScaleBytes;  // bytes one quadrant's copy lands per page
constexpr int kQBoxBytes = kRowsPerCta * 64 * 2;   // 128 query rows x 64 latent bf16, 16 KiB
constexpr int kQRopeBox = kRowsPerCta * 32 * 2;    // 32 RoPE columns of 128 query rows, 64-byte swizzle
// Shared memory of the two modes of the kernel:
//   pair (one latent group): a stage holds this CTA's latent half and its
//        32 RoPE columns of a page; send slots (2) | receive slots (2) | the
//        RoPE query tile (128 rows x this CTA's 32 columns) | DecodeShared.
//   solo (2, 4 or 8 groups): a stage holds this CTA's latent half and all
//        64 RoPE columns; P slots (2) | the RoPE query tile (128 rows x 64
//        columns, two boxes) | DecodeShared.
// FP8 cache (kFp8): a stage holds only the dequantised latent half (f16);
// the page's raw codes and scales land in one of two raw slots (freed by the
// dequantising warp once read) and its RoPE columns in a ring of their own
// (freed by the QK MMAs), both ahead of the stage:
//   f16 stages (3) | RoPE ring (3) | raw slots (2) | as above from the send slots on.
constexpr int kStagesFp8 = 3;
constexpr int kRawSlots = 2;
constexpr int kRawBoxBytes = kPage * 64;                 // 64 tokens x 64 codes, unswizzled, 4 KiB
constexpr int kRawScaleBytes = kPage * 16;               // 64 tokens x 4 fp32 scales, 1 KiB
constexpr int kRawSlotBytes = 4 * kRawBoxBytes + kRawScaleBytes;
template <bool kSolo, bool kFp8>
struct Layout {
  static constexpr int kNStages = kFp8 ? kStagesFp8 : kStages;
  static constexpr int kRopeBoxes = kSolo ? 2 : 1;
  static constexpr int kRopeBytes = kRopeBoxes * kRopeBoxBytes;  // a page's RoPE columns of this CTA
  static constexpr int kStageBytes = 4 * kBoxBytes + (kFp8 ? 0 : kRopeBytes);
  static constexpr int kRopeRingOff = kNStages * kStageBytes;
  static constexpr int kRawOff = kRopeRingOff + (kFp8 ? kNStages * kRopeBytes : 0);
  static constexpr int kXOff = kRawOff + (kFp8 ? kRawSlots * kRawSlotBytes : 0);  // send slots (pair), P slots (solo)
  static constexpr int kRecvOff = kSolo ? kXOff : kXOff + 2 * kXSlot;     // P is written here
  static constexpr int kQRopeOff = kXOff + (kSolo ? 2 : 4) * kXSlot;
  static constexpr int kQRopeBytes = kRopeBoxes * kQRopeBox;
  static constexpr int kSmemShared = kQRopeOff + kQRopeBytes;
  // the RoPE columns of the page in stage st
  static constexpr int rope_off(int st) { return kFp8 ? kRopeRingOff + st * kRopeBytes : st * kStageBytes + 4 * kBoxBytes; }
  static_assert(kStageBytes % 1024 == 0 && kXSlot % 1024 == 0 && kQRopeOff % 1024 == 0 && kRawOff % 1024 == 0 &&
                    kRawSlotBytes % 1024 == 0 && kRopeBytes % 512 == 0,
                "swizzled tiles need aligned bases");
};
static_assert(4 * kQBoxBytes == 4 * kXSlot, "the first query's latent half fills the four exchange slots");
// warps 0-7: softmax warps (TMEM lane quadrant w & 3, key half w >> 2: 32
// keys of every page, 128 columns of O, 64 columns of Q); then, in pair
// mode, warps 8-11: exchange warps (one per quadrant, a whole score row per
// thread); then the TMA producer and the QK and P.V issuers (warps 12-14 in
// pair mode, 8-10 in solo mode, which exchanges nothing); with an FP8 cache
// one more warp dequantises the pages.  A warp's SM sub-partition is its
// index mod 4, and the TMEM quadrant of the softmax and exchange warps fixes
// theirs; in pair mode over a bf16 cache the TMA producer runs as warp 15
// (sub-partition 3, whose softmax warps have the most slack; measured 1 %
// faster on the long and speculative workloads) and warp 12 idles.  15 or
// 16 warps leave 128 registers a thread (four warps share an SM
// sub-partition's 64K); the 11 or 12 of solo mode leave 168.
constexpr int kSWarps = 8, kXWarps = 4;
constexpr int kSoftmaxThreads = 32 * kSWarps, kXThreads = 32 * kXWarps;
template <bool kSolo, bool kFp8>
struct Roles {
  static constexpr int kX = kSolo ? 0 : kXWarps;  // exchange warps
  static constexpr bool kTmaLast = !kSolo && !kFp8;
  static constexpr int kTma = kTmaLast ? 15 : kSWarps + kX, kMma = kSWarps + kX + 1, kPv = kMma + 1;
  static constexpr int kIdle = kTmaLast ? kSWarps + kX : -1;
  static constexpr int kDq = kFp8 ? kPv + 1 : -1;  // dequantising warp
  static constexpr int kThreads = kTmaLast ? 512 : 32 * (kPv + 1 + (kFp8 ? 1 : 0));
};
static_assert(kPlanInKernelMaxB <= Roles<false, false>::kThreads &&
                  kPlanInKernelMaxBSolo <= Roles<true, false>::kThreads,
              "the in-kernel plan takes one thread per sequence");
// named barriers 1..4: the two softmax warps of a quadrant
constexpr uint32_t kBarPair0 = 1;
constexpr int kPlanWarpMaxB = 32;  // up to this batch one warp plans (lane = sequence)
// tensor memory columns: O (256) | Q latent half (128, bf16 pairs) | two
// score buffers (64 each)
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384, kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: defer O rescaling up to 2^8

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Copy `bytes` of this CTA's shared memory into another CTA of the cluster;
// completion is counted in bytes on the destination CTA's mbarrier.  The
// copies of one thread form bulk groups, so it can wait until their source
// has been read (bulk_wait_read_all).
__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst_cluster), "r"(src), "r"(bytes), "r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Partial scores cross the pair as 16-bit fixed point with a power-of-two
// scale per row: q = round(x * 2^k), k chosen so that the row's largest |x|
// maps below 2^14.  The absolute error of every key is then at most 2^-14 of
// the row's largest |partial|, about 8 times below that of fp16 at the same
// size, and independent of where the key sits in the row.  The rounding
// uses the float adder: x * 2^k + (1.5 * 2^23 + 2^15) holds q + 2^15 in its
// low 16 mantissa bits, and a byte permute puts those bits back under the
// same exponent on the receiving side, so both directions stay on full-rate
// FMA and integer pipes instead of the conversion unit.
constexpr float kRoundMagic = 12615680.0f;      // 1.5 * 2^23 + 2^15
constexpr uint32_t kRoundMagicHigh = 0x4B400000u;  // the top 16 bits of its encoding (low bits vary)
__device__ __forceinline__ int row_scale_exp(float maxabs) {
  const int e = (int)((__float_as_uint(maxabs) >> 23) & 0xffu) - 127;  // floor(log2 maxabs) (normal numbers)
  const int k = 13 - e;
  return k < -100 ? -100 : (k > 100 ? 100 : k);  // zero or tiny rows: any scale will do
}
__device__ __forceinline__ float exp2_int(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }
// two values already multiplied by 2^k -> two rounded 16-bit codes (q + 2^15)
__device__ __forceinline__ uint32_t pack_fixed16x2(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo + kRoundMagic), __float_as_uint(hi + kRoundMagic), 0x5410);
}
__device__ __forceinline__ float2 unpack_fixed16x2(uint32_t w) {
  return make_float2(__uint_as_float(__byte_perm(w, kRoundMagicHigh, 0x7610)) - kRoundMagic,
                     __uint_as_float(__byte_perm(w, kRoundMagicHigh, 0x7632)) - kRoundMagic);
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// largest of 32 values (three-input maxima)
__device__ __forceinline__ float max32(const float (&x)[32]) {
  float m[11];
#pragma unroll
  for (int j = 0; j < 10; ++j) m[j] = fmax3(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
  m[10] = fmaxf(x[30], x[31]);
  const float a = fmax3(m[0], m[1], m[2]), b = fmax3(m[3], m[4], m[5]), c = fmax3(m[6], m[7], m[8]);
  return fmaxf(fmax3(a, b, c), fmaxf(m[9], m[10]));
}
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Named barrier `id` over `n` threads with an AND vote: every thread learns
// whether all of them are still ok (so none is left waiting alone).
__device__ __forceinline__ bool bar_red_and_n(bool ok, uint32_t id, uint32_t n) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(r) : "r"((uint32_t)ok), "r"(id), "r"(n) : "memory");
  return r != 0;
}

__device__ __forceinline__ void set_status(WsHeader* ws, int code) {
  atomicCAS(&ws->status, 0, code);
}

// FP8 cache, the dequantising warp: lane j's 16 codes of each of the eight
// 512-byte sweeps of raw box q (rows 8*it + j/4, codes 16*(j%4) ...).
__device__ __forceinline__ void load_codes(uint32_t raw, int q, int lane, uint4 (&w)[8]) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const uint32_t a = raw + q * kRawBoxBytes + it * 512 + lane * 16;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w[it].x), "=r"(w[it].y), "=r"(w[it].z), "=r"(w[it].w) : "r"(a));
  }
}
// ... and the scale of 128-column block `blk` of those eight rows
__device__ __forceinline__ void load_scales(uint32_t raw, int blk, int lane, float (&sc)[8]) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const uint32_t a = raw + 4 * kRawBoxBytes + (it * 8 + (lane >> 2)) * 16 + 4 * blk;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sc[it]) : "r"(a));
  }
}
// Box q's codes (loaded by load_codes) times their rows' scales (sc[it],
// the box's block) as f16 into the stage, in the 128-byte swizzled K-major
// layout.  Returns true if a scale is neither 0 nor a value in [2^-15, 2^7]
// (its products may leave the f16 range).
__device__ __forceinline__ bool dequant_box(const uint4 (&w)[8], const float (&sc)[8], int q, uint32_t dst, int lane) {
  bool bad = false;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = it * 8 + (lane >> 2);
    const float s = sc[it];
    bad |= !(s == 0.f || (s >= 0x1p-15f && s <= 0x1p7f));
    const uint32_t s2 = pack_f16x2(s, s);
    const uint32_t cw[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t lo, hi;
      e4m3x4_to_f16x2x2(cw[k], lo, hi);
      h[2 * k] = mul_f16x2(lo, s2);
      h[2 * k + 1] = mul_f16x2(hi, s2);
    }
    const uint32_t drow = dst + q * kBoxBytes + row * 128;
    const int c0 = 2 * (lane & 3);
    st_shared_v4(drow + ((c0 ^ (row & 7)) << 4), h[0], h[1], h[2], h[3]);
    st_shared_v4(drow + (((c0 + 1) ^ (row & 7)) << 4), h[4], h[5], h[6], h[7]);
  }
  return bad;
}

// A query chunk (64 bf16) to f16 for the f16 MMAs of an FP8 cache; true if
// a value lies beyond the f16 range (it becomes infinite).
__device__ __forceinline__ bool query_to_f16(uint32_t (&w)[32]) {
  bool over = false;
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const uint32_t h = bf16x2_to_f16x2(w[k]);
    over |= ((h & 0x7fffu) == 0x7c00u) || ((h & 0x7fff0000u) == 0x7c000000u);
    w[k] = h;
  }
  return over;
}

// Shared state of one decode CTA (at the end of dynamic shared memory).
// Per score buffer / receive slot b (page parity):
//   s_full   QK(p) wrote the own partial scores into S_b
//   xfull    [b][quadrant]: the peer's 16-bit partial of that quadrant's
//            32 rows and their scales landed (receive slot b, xscale_recv)
//   s_free   the exchange and softmax warps read S_b (the next QK may
//            overwrite it)
//   p_full   P(p) is in receive slot b
//   o_done   P.V of page p is done
//   can_send the peer's P.V of page p is done: its receive slot b is free
//            again (a remote arrive from the peer's P.V thread); phase 0
//            instead says the peer's first query left its slots
// Per segment:
//   q_lat    the first segment's query (latent half in the receive slots,
//            RoPE half in its tile) landed
//   q_full   a segment's latent query is in tensor memory
//   q_tma    a later segment's RoPE query tile landed
//   drain    [QK, P.V]: every MMA the issuing thread started is done
//            (teardown after an abort)
// Per page, FP8 cache only (stage st = page % 3, raw slot = page % 2):
//   raw_full   the page's codes, scales and RoPE columns landed
//   raw_empty  the dequantising warp read the raw slot
//   full[st]   the dequantised latent is in stage st (an arrival of that warp)
//   rope_empty QK of the page is done: its RoPE ring slot is free
struct DecodeShared {
  float xscale_send[2][kRowsPerCta];  // 2^-k of each row's 16-bit partial: ours (copied to the peer)
  float xscale_recv[2][kRowsPerCta];  // and the peer's
  uint64_t full[kStages], empty[kStages];
  uint64_t raw_full[kRawSlots], raw_empty[kRawSlots], rope_empty[kStagesFp8];  // FP8 cache only
  uint64_t q_full, q_tma, q_lat, drain[2];
  uint64_t never;                // testing: a barrier nothing completes (see DecodeArgs::stall_page)
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2], can_send[2];
  uint64_t xfull[2][4];
  float red[2][2][kRowsPerCta];  // [parity][key half][row]: partial row maxima (row sums at a segment's end)
  UnitRec rec;                   // this CTA's work unit
  uint32_t tmem;
  int abort;
  int peer_sent[4];              // pages the peer's exchange warp of each quadrant sent here (teardown)
  int lens[kPlanInKernelMaxB];   // validated sequence lengths (in-kernel plan)
  int16_t qsrc[kSoftmaxThreads][2];  // softmax thread's q_cat column of each latent chunk (-1: zeros)
};

// All shared memory is dynamic: stage ring, exchange slots, then the small state.
template <bool kSolo, bool kFp8>
constexpr int decode_smem() {
  return Layout<kSolo, kFp8>::kSmemShared + (int)((sizeof(DecodeShared) + 15) & ~size_t(15));
}
static_assert(decode_smem<false, false>() <= 232448 && decode_smem<true, false>() <= 232448 &&
                  decode_smem<false, true>() <= 232448 && decode_smem<true, true>() <= 232448,
              "decode kernel exceeds 227 KiB of shared memory");

__device__ __forceinline__ int clamp_len(int n, int lo, int hi) { return n < lo ? lo : (n > hi ? hi : n); }
// units given to a sequence of np pages by the sequence-aligned split
__device__ __forceinline__ int aligned_units(int np, int units, int total) {
  return min(np, max(1, (int)(((long long)units * np) / total)));
}

// Walks the (sequence, page range) segments of one work unit from its
// UnitRec, reading page counts from seq_lens (validated lengths).
// Lengths come from shared memory (validated by the in-kernel plan) or,
// when the plan kernel split the work, from seq_lens (clamped here).
struct SegIter {
  int b, o, start, end, bias;
  const int* lens;
  bool raw;
  __device__ void init(const UnitRec& r, const int* l, bool clamp) {
    b = r.b; o = r.o; start = r.start; end = r.end; bias = r.bias;
    lens = l; raw = clamp;
  }
  __device__ int slot(int sb) const { return sb + bias; }
  __device__ int len(const DecodeArgs& a, int sb) const {
    return raw ? clamp_len(lens[sb], a.Lq > 1 ? a.Lq : 1, a.max_pages * kPage) : lens[sb];
  }
  // Next non-empty segment: sequence sb, pages [pa, pb) of that sequence.
  __device__ bool next(const DecodeArgs& a, int& sb, int& pa, int& pb) {
    while (b < a.B && start < end) {
      const int o0 = o;
      if (o0 >= end) break;
      const int o1 = o0 + (len(a, b) + kPage - 1) / kPage;
      const int aa = max(start, o0), e = min(end, o1);
      const int cur = b++;
      o = o1;
      if (aa < e) {
        sb = cur;
        pa = aa - o0;
        pb = e - o0;
        return true;
      }
    }
    return false;
  }
};

// One unit's pages in order: page i of sequence sb, in the segment [pa, pb).
struct PageCursor {
  SegIter it;
  int sb, pa, pb, i;
  bool valid;
  __device__ void init(const UnitRec& r, const DecodeArgs& a, const int* l, bool clamp) {
    it.init(r, l, clamp);
    valid = it.next(a, sb, pa, pb);
    i = pa;
  }
  __device__ void advance(const DecodeArgs& a) {
    if (++i >= pb) {
      valid = it.next(a, sb, pa, pb);
      i = pa;
    }
  }
  __device__ bool seg_first() const { return i == pa; }
  __device__ bool seg_last() const { return i == pb - 1; }
};

// ---- small block-wide helpers (all threads of the block call them)
__device__ __forceinline__ int block_reduce_max(int v, int* scratch) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int w = threadIdx.x < (int)(blockDim.x >> 5) ? scratch[threadIdx.x] : INT_MIN;
    for (int o = 16; o > 0; o >>= 1) w = max(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (threadIdx.x == 0) scratch[32] = w;
  }
  __syncthreads();
  const int r = scratch[32];
  __syncthreads();
  return r;
}
// inclusive block scan of one value per thread; *total receives the sum
__device__ __forceinline__ int block_scan_incl(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  if (lane == 31) scratch[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? scratch[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += x;
    }
    if (lane < nw) scratch[lane] = t;
    if (lane == nw - 1) scratch[32] = t;
  }
  __syncthreads();
  if (w > 0) v += scratch[w - 1];
  *total = scratch[32];
  __syncthreads();
  return v;
}

constexpr int kSwitchPages = 4;  // cost of a sequence switch inside a unit, in pages

// The split of mla_decode_paged's work, computed by one block with one
// thread per sequence (B <= blockDim.x): validated lengths, page prefix sums,
// the cheaper of the balanced and sequence-aligned splits (see plan_kernel),
// and this unit's UnitRec.  `writer` also stores the per-sequence slot
// ranges and the header for the combine kernel.  scr: >= 3*B + 3 ints of
// shared scratch; red: 33 ints.
__device__ void plan_in_block(const DecodeArgs& a, int unit, bool writer, int* scr, int* red, int* lens_s,
                              UnitRec* out) {
  const int B = a.B, units = a.units, tid = threadIdx.x;
  const WsView v = ws_view(a.ws, B);
  int* off_s = scr;            // [B+1]
  int* u0_s = scr + B + 1;     // [B+1]
  const int lo = a.Lq > 1 ? a.Lq : 1, hi = a.max_pages * kPage;
  int np = 0;
  if (tid < B) {
    const int n0 = a.seq_lens[tid];
    const int n = clamp_len(n0, lo, hi);
    if (writer) {
      if (n != n0) set_status(a.ws, MLA_ERR_BAD_SEQLEN);
      v.nlen[tid] = n;
    }
    lens_s[tid] = n;
    np = (n + kPage - 1) / kPage;
  }
  int total = 0;
  const int incl = block_scan_incl(np, red, &total);
  if (tid < B) off_s[tid] = incl - np;
  if (tid == 0) off_s[B] = total;
  __syncthreads();
  const int chunk = total > 0 ? (total + units - 1) / units : 1;

  int segs = 0;  // balanced split: most sequences one unit touches
  for (int k = tid; k < units; k += blockDim.x) {
    const int st = min(k * chunk, total), en = min(st + chunk, total);
    if (st < en) {
      int l0 = 0, h0 = B - 1, l1 = 0, h1 = B - 1;
      while (l0 < h0) { const int m = (l0 + h0 + 1) >> 1; if (off_s[m] <= st) l0 = m; else h0 = m - 1; }
      while (l1 < h1) { const int m = (l1 + h1 + 1) >> 1; if (off_s[m] <= en - 1) l1 = m; else h1 = m - 1; }
      segs = max(segs, l1 - l0 + 1);
    }
  }
  segs = block_reduce_max(segs, red);
  const int cost_bal = chunk + kSwitchPages * (segs - 1);

  const bool feasible = B <= units && total > 0;
  int u = 0, worst = 0, used = 0;
  if (feasible && tid < B) {
    u = aligned_units(np, units, total);
    worst = (np + u - 1) / u;
  }
  const int uincl = block_scan_incl(u, red, &used);
  if (tid < B) u0_s[tid] = uincl - u;
  worst = block_reduce_max(worst, red);
  const int cost_al = (feasible && used <= units) ? worst : INT_MAX;
  const int mode = cost_al <= cost_bal ? 1 : 0;

  if (tid == 0) {
    UnitRec rec{0, 0, 0, 0, 0};
    if (mode == 1) {
      if (unit < used) {
        int l0 = 0, h0 = B - 1;
        while (l0 < h0) { const int m = (l0 + h0 + 1) >> 1; if (u0_s[m] <= unit) l0 = m; else h0 = m - 1; }
        const int nb = off_s[l0 + 1] - off_s[l0], ub = aligned_units(nb, units, total), j = unit - u0_s[l0];
        rec = UnitRec{l0, 0, (int)(((long long)j * nb) / ub), (int)(((long long)(j + 1) * nb) / ub), unit - l0};
      }
    } else {
      const int st = min(unit * chunk, total), en = min(st + chunk, total);
      int l0 = 0, h0 = B - 1;
      while (l0 < h0) { const int m = (l0 + h0 + 1) >> 1; if (off_s[m] <= st) l0 = m; else h0 = m - 1; }
      rec = UnitRec{l0, off_s[l0], st, en, unit};
    }
    *out = rec;
  }
  if (writer) {
    if (tid < B) {
      v.off[tid] = off_s[tid];
      if (mode == 1) {
        v.slot0[tid] = u0_s[tid];
        v.nslot[tid] = u;
      } else {
        const int o0 = off_s[tid], kf = o0 / chunk, kl = (o0 + np - 1) / chunk;
        v.slot0[tid] = tid + kf;
        v.nslot[tid] = kl - kf + 1;
      }
    }
    if (tid == 0) {
      v.off[B] = total;
      a.ws->total = total;
      a.ws->chunk = chunk;
      a.ws->units = units;
      a.ws->B = B;
      a.ws->mode = mode;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ int warp_scan_incl(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  return v;
}

// plan_in_block's split for B <= 32, computed by one warp (lane = sequence)
// with shuffles and votes instead of block-wide barriers.  The balanced
// split's widest unit is found by counting, per unit, the sequences that
// start strictly inside it (the unit touches one more sequence than that).
// n0: seq_lens[lane] (lanes < B), loaded by the caller ahead of time.
__device__ void plan_in_warp(const DecodeArgs& a, int unit, bool writer, int n0, int* lens_s, UnitRec* out) {
  const unsigned full = 0xffffffffu;
  const int B = a.B, units = a.units, lane = threadIdx.x & 31;
  const WsView v = ws_view(a.ws, B);
  const int lo = a.Lq > 1 ? a.Lq : 1, hi = a.max_pages * kPage;
  const bool act = lane < B;
  int np = 0;
  if (act) {
    const int n = clamp_len(n0, lo, hi);
    if (writer) {
      if (n != n0) set_status(a.ws, MLA_ERR_BAD_SEQLEN);
      v.nlen[lane] = n;
    }
    lens_s[lane] = n;
    np = (n + kPage - 1) / kPage;
  }
  const int incl = warp_scan_incl(np);
  const int total = __shfl_sync(full, incl, 31);
  const int off = incl - np;
  const int chunk = total > 0 ? (total + units - 1) / units : 1;

  const bool inner = act && off % chunk != 0;  // sequence starts inside unit off / chunk
  const int key = inner ? off / chunk : -1 - lane;
  const unsigned same = __match_any_sync(full, key);
  const int segs = 1 + (int)__reduce_max_sync(full, inner ? (unsigned)__popc(same) : 0u);
  const int cost_bal = chunk + kSwitchPages * (segs - 1);

  const bool feasible = B <= units && total > 0;
  int u = 0, worst = 0;
  if (feasible && act) {
    u = aligned_units(np, units, total);
    worst = (np + u - 1) / u;
  }
  const int uincl = warp_scan_incl(u);
  const int used = __shfl_sync(full, uincl, 31);
  const int u0 = uincl - u;
  worst = (int)__reduce_max_sync(full, (unsigned)worst);
  const int cost_al = (feasible && used <= units) ? worst : INT_MAX;
  const int mode = cost_al <= cost_bal ? 1 : 0;

  UnitRec rec{0, 0, 0, 0, 0};
  if (mode == 1) {
    const unsigned m = __ballot_sync(full, act && u0 <= unit);  // lane 0 always: u0 = 0
    const int l0 = 31 - __clz(m);
    const int nb = __shfl_sync(full, np, l0), ub = __shfl_sync(full, u, l0), j = unit - __shfl_sync(full, u0, l0);
    if (unit < used)
      rec = UnitRec{l0, 0, (int)(((long long)j * nb) / ub), (int)(((long long)(j + 1) * nb) / ub), unit - l0};
  } else {
    const int st = min(unit * chunk, total), en = min(st + chunk, total);
    const unsigned m = __ballot_sync(full, act && off <= st);
    const int l0 = 31 - __clz(m);
    rec = UnitRec{l0, __shfl_sync(full, off, l0), st, en, unit};
  }
  if (lane == 0) *out = rec;
  if (writer) {
    if (act) {
      v.off[lane] = off;
      if (mode == 1) {
        v.slot0[lane] = u0;
        v.nslot[lane] = u;
      } else {
        const int kf = off / chunk, kl = (off + np - 1) / chunk;
        v.slot0[lane] = lane + kf;
        v.nslot[lane] = kl - kf + 1;
      }
    }
    if (lane == 0) {
      v.off[B] = total;
      a.ws->total = total;
      a.ws->chunk = chunk;
      a.ws->units = units;
      a.ws->B = B;
      a.ws->mode = mode;
    }
  }
  __syncwarp();
}

// kSolo: 2, 4 or 8 latent groups.  Every group latent lies inside one
// latent half, so CTA r of the pair serves the heads whose group latent is
// in its half (heads r*H/2 .. (r+1)*H/2 - 1) with their whole scores: it
// loads all 64 RoPE columns and exchanges nothing with the peer.  Its
// query rows are (l, h) for those heads, l-major.
template <bool kSolo, bool kFp8>
__global__ void __launch_bounds__(Roles<kSolo, kFp8>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_cache, const __grid_constant__ CUtensorMap tm_rope,
                  const __grid_constant__ CUtensorMap tm_qrope, const __grid_constant__ CUtensorMap tm_qlat,
                  const __grid_constant__ CUtensorMap tm_scale, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  using L = Layout<kSolo, kFp8>;
  using R = Roles<kSolo, kFp8>;
  constexpr int kStageBytes = L::kStageBytes;
  constexpr int NS = L::kNStages;
  const uint32_t xsend = smem_u32(smem + L::kXOff);     // send slots 0 and 1 (pair)
  const uint32_t xrecv = smem_u32(smem + L::kRecvOff);  // receive slots (pair), P slots (solo)
  const uint32_t qrope = smem_u32(smem + L::kQRopeOff);
  DecodeShared& sh = *reinterpret_cast<DecodeShared*>(smem + L::kSmemShared);
  constexpr int kXW = R::kX;
  constexpr int kTmaWarp = R::kTma, kMmaWarp = R::kMma, kPvWarp = R::kPv, kDqWarp = R::kDq;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 128-byte-swizzled tiles need a 1024-byte aligned base; the whole cluster
  // sees the same layout, so every CTA takes this exit together.
  if (smem_u32(smem) & 1023u) {
    griddep_wait();
    if (threadIdx.x == 0) set_status(a.ws, MLA_ERR_UNSUPPORTED);
    return;
  }
  const uint32_t crank = cluster_ctarank();
  const uint32_t r = crank & 1u;         // latent half owned by this CTA
  const uint32_t rg = crank >> 1;        // 128-row block of the query rows
  const uint32_t peer = crank ^ 1u;
  const int unit = (int)cluster_id_x();
  WsHeader* ws = a.ws;
  const uint64_t lim = a.wait_ns;        // limit of every pipeline wait

  auto bar = [](uint64_t& x) { return smem_u32(&x); };
  const bool warp_plan = a.plan_in_kernel && a.B <= kPlanWarpMaxB;

  // Warp 0 (the planning warp for small batches) waits for the kernel
  // before and requests the sequence lengths at once, so their load
  // overlaps the set-up below.  The TMA warp pulls this CTA's share of the
  // block table into L2 (a prefetch cannot return stale data, so it may
  // precede the wait).
  int n_pre = 0;
  if (warp == 0 && warp_plan) {
    griddep_wait();
    if (lane < a.B) n_pre = a.seq_lens[lane];
  } else if (warp == kTmaWarp) {
    const size_t lines = ((size_t)a.B * a.max_pages * 4 + 127) / 128;
    const size_t ctas = (size_t)gridDim.x, per = (lines + ctas - 1) / ctas;
    const char* tb = reinterpret_cast<const char*>(a.block_table);
    for (size_t k = lane; k < per && k < 256; k += 32) {
      const size_t line = (size_t)blockIdx.x * per + k;
      if (line < lines) asm volatile("prefetch.global.L2 [%0];" ::"l"(tb + line * 128));
    }
  }
  if (threadIdx.x == kTmaWarp * 32) {
    sh.abort = 0;
    for (int q = 0; q < 4; ++q) sh.peer_sent[q] = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(sh.full[s]), 1);
      mbar_init(bar(sh.empty[s]), 1);
    }
    if constexpr (kFp8) {
      for (int s = 0; s < kRawSlots; ++s) {
        mbar_init(bar(sh.raw_full[s]), 1);
        mbar_init(bar(sh.raw_empty[s]), 1);
      }
      for (int s = 0; s < NS; ++s) mbar_init(bar(sh.rope_empty[s]), 1);
    }
    mbar_init(bar(sh.q_full), kSoftmaxThreads);
    mbar_init(bar(sh.q_tma), 1);
    mbar_init(bar(sh.q_lat), 1);
    mbar_init(bar(sh.drain[0]), 1);
    mbar_init(bar(sh.drain[1]), 1);
    mbar_init(bar(sh.never), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(sh.s_full[s]), 1);
      mbar_init(bar(sh.s_free[s]), kSoftmaxThreads + (kSolo ? 0 : kXThreads));
      mbar_init(bar(sh.p_full[s]), kSoftmaxThreads);
      mbar_init(bar(sh.o_done[s]), 1);
      mbar_init(bar(sh.can_send[s]), 1);  // one remote arrival from the peer
      for (int q = 0; q < 4; ++q) mbar_init(bar(sh.xfull[s][q]), 1);  // armed, completed by the peer's stores
    }
    fence_mbar_init();
    for (int s = 0; s < 2; ++s)
      for (int q = 0; q < 4; ++q) mbar_arrive_expect_tx(bar(sh.xfull[s][q]), kXQuadTx);
    tma_prefetch_desc(&tm_cache);
    tma_prefetch_desc(&tm_rope);
    tma_prefetch_desc(&tm_qrope);
    tma_prefetch_desc(&tm_qlat);
    if constexpr (kFp8) tma_prefetch_desc(&tm_scale);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sh.tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // The peer's barriers must be initialised before any remote arrive or
  // copy: arrive on the cluster barrier now (relaxed: the initialisation
  // fence above already orders the barrier set-up), wait after the plan.
  cluster_arrive_relaxed();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;
  volatile int* abort = &sh.abort;
  // set-up above overlaps the kernel before; global memory only from here on
  griddep_wait();
  griddep_launch_dependents();

  // the work split: computed here (by one warp for small batches, else by
  // the whole block with the still unused exchange slots as scratch), or
  // read from the plan kernel's records
  if (a.plan_in_kernel && a.B <= kPlanWarpMaxB) {
    if (warp == 0) plan_in_warp(a, unit, unit == 0 && crank == 0, n_pre, sh.lens, &sh.rec);
  } else if (a.plan_in_kernel) {
    int* scratch = reinterpret_cast<int*>(smem + L::kXOff);
    plan_in_block(a, unit, unit == 0 && crank == 0, scratch, scratch + 3 * a.B + 8, sh.lens, &sh.rec);
  } else if (threadIdx.x == 0) {
    sh.rec = ws_view(ws, a.B).rec[unit];
  }
  fence_proxy_async();  // the plan's scratch writes come before the query copies into the same slots
  __syncthreads();
  cluster_wait();
  const int* lens = a.plan_in_kernel ? sh.lens : a.seq_lens;  // where the page walkers read lengths
  const bool lens_raw = !a.plan_in_kernel;

  // A wait that gives up stops both CTAs of the pair.
  const uint32_t peer_abort = mapa(smem_u32(&sh.abort), peer);
  auto fail = [&]() {
    *abort = 1;
    st_cluster_u32(peer_abort, 1u);
    set_status(ws, MLA_ERR_TIMEOUT);
  };
  // What this thread started and the teardown must see finished.
  uint32_t issued = 0;  // TMA producer: pages whose copies were issued
  uint32_t nq_tma = 0;  // thread 0: RoPE query tiles loaded by TMA for later segments
  int sent = 0;         // exchange warps: pages copied to the peer
  bool bad_scale = false;  // FP8: a scale outside the exact f16 range was read

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp walks the unit's pages (lane 0 issues the copies); the
    // block-table entries of up to 32 pages come in with one coalesced load.
    {
      const uint32_t bytes = kStageBytes;
      const uint64_t policy = l2_policy_evict_first();
      SegIter it;
      it.init(sh.rec, lens, lens_raw);
      int sb, pa, pb;
      bool ok = true;
      bool first_seg = true;
      while (ok && it.next(a, sb, pa, pb)) {
        const int32_t* bt = a.block_table + (size_t)sb * a.max_pages;
        if (kSolo && !first_seg) {
          // the query rows of this segment's sequence into L2, well before
          // the softmax warps load them at the end of the segment before
          const char* q0 = reinterpret_cast<const char*>(a.q_cat + (size_t)sb * a.Lq * a.H * (a.d_g + kDr));
          const int lines = (a.Lq * a.H * (a.d_g + kDr) * 2 + 127) / 128;
          for (int k = lane; k < lines; k += 32) asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(q0 + 128 * k));
        }
        first_seg = false;
        for (int c0 = pa; ok && c0 < pb; c0 += 32) {
          const int nc = min(32, pb - c0);
          const int mine = lane < nc ? bt[c0 + lane] : 0;
          for (int j = 0; j < nc; ++j) {
            const uint32_t pc = issued;
            const int st = pc % NS;
            if constexpr (kFp8) {  // the raw slot read by the dequantising warp, the RoPE slot by QK
              if (pc >= (uint32_t)kRawSlots)
                ok = mbar_wait(bar(sh.raw_empty[pc % kRawSlots]), ((pc / kRawSlots) - 1) & 1, abort, lim);
              if (ok && pc >= (uint32_t)NS) ok = mbar_wait(bar(sh.rope_empty[st]), ((pc / NS) - 1) & 1, abort, lim);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
            } else if (pc >= (uint32_t)NS) {
              ok = mbar_wait(bar(sh.empty[st]), ((pc / NS) - 1) & 1, abort, lim);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
            }
            int page = __shfl_sync(0xffffffffu, mine, j);
            if (page < 0 || page >= a.num_pages) {  // never dereferenced: clamped and reported
              if (lane == 0) set_status(ws, MLA_ERR_BAD_TABLE);
              page = 0;
            }
            if (lane == 0) {
              if (!kSolo && pc == 0) {  // the first segment's query, ahead of its first page
                // latent boxes of 64 columns: this CTA's half of the latent
                // (one group), or the first columns of each row's own
                // group latent (several groups)
                const int qy = sb * a.Lq * a.H + (int)rg * kRowsPerCta;
                const int qx = a.G == 1 ? (int)r * 256 : 0;
                const int nbox = a.G == 1 ? 4 : min(a.d_g, 256) / 64;
                mbar_arrive_expect_tx(bar(sh.q_lat), nbox * kQBoxBytes + kQRopeBox);
                for (int q = 0; q < nbox; ++q)
                  tma_load_2d(xsend + q * kQBoxBytes, &tm_qlat, bar(sh.q_lat), qx + 64 * q, qy);
                tma_load_2d(qrope, &tm_qrope, bar(sh.q_lat), a.d_g + 32 * (int)r, qy);
              }
              if constexpr (kFp8) {
                // this CTA's 256 codes of each row (four 64-byte boxes), the
                // rows' four scales, and the RoPE columns into the ring slot
                const uint32_t raw = smem_u32(smem + L::kRawOff + (pc % kRawSlots) * kRawSlotBytes);
                const uint32_t rb = bar(sh.raw_full[pc % kRawSlots]);
                mbar_arrive_expect_tx(rb, kRawSlotBytes + L::kRopeBytes);
                for (int q = 0; q < 4; ++q)
                  tma_load_2d_hint(raw + q * kRawBoxBytes, &tm_cache, rb, (int)(r * 256 + q * 64), page * kPage,
                                   policy);
                tma_load_2d_hint(raw + 4 * kRawBoxBytes, &tm_scale, rb, kFp8ScaleByte / 4, page * kPage, policy);
                for (int q = 0; q < L::kRopeBoxes; ++q)
                  tma_load_2d_hint(smem_u32(smem + L::rope_off(st)) + q * kRopeBoxBytes, &tm_rope, rb,
                                   kFp8RopeByte / 2 + 32 * (kSolo ? q : (int)r), page * kPage, policy);
              } else {
                const uint32_t dst = smem_u32(stages + st * kStageBytes);
                mbar_arrive_expect_tx(bar(sh.full[st]), bytes);
                for (int q = 0; q < 4; ++q)  // this CTA's latent half
                  tma_load_2d_hint(dst + q * kBoxBytes, &tm_cache, bar(sh.full[st]), (int)(r * 256 + q * 64),
                                   page * kPage, policy);
                // this CTA's 32 RoPE columns (all 64 in solo mode)
                for (int q = 0; q < L::kRopeBoxes; ++q)
                  tma_load_2d_hint(dst + 4 * kBoxBytes + q * kRopeBoxBytes, &tm_rope, bar(sh.full[st]),
                                   kDc + 32 * (kSolo ? q : (int)r), page * kPage, policy);
              }
            }
            ++issued;
          }
        }
      }
      if (!ok && lane == 0) fail();
    }
    __syncwarp();  // reconverge before the CTA-wide barrier of the teardown
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ QK issuer
    // Per page p in score buffer b = p & 1:
    //   QK(p):  S_b = Q . K^T over this CTA's columns               (this warp)
    //   PV(p):  O  += P (receive slot b, written by the softmax) . V (next warp)
    // Two issuing threads keep the tensor pipe fed: QKs wait only for their
    // page and score buffer, P.Vs for the softmax.  Every dependence between
    // the streams goes through an mbarrier.
    if (lane == 0) {
      // the latent K steps in f16 when the cache is FP8 (dequantised tile,
      // f16 query); the RoPE K steps always in bf16; one fp32 accumulator
      constexpr uint32_t idesc_qk = idesc_bf16(128, 64, false, false);
      constexpr uint32_t idesc_qk_lat = kFp8 ? idesc_f16(128, 64, false, false) : idesc_qk;
      const uint64_t qr0 = sdesc_sw64(qrope, 512);
      PageCursor c;
      c.init(sh.rec, a, lens, lens_raw);
      uint32_t pc = 0, qc = 0;
      bool ok = true;
      while (ok && c.valid) {
        if (c.seg_first()) {  // the segment's query (loaded after every QK before it finished)
          if (!(ok = mbar_wait(bar(sh.q_full), qc & 1, abort, lim))) break;
          // the RoPE query tile by TMA: every segment in solo mode, later ones in pair mode
          const uint32_t nt = kSolo ? qc : qc - 1;
          if ((kSolo || qc > 0) && !(ok = mbar_wait(bar(sh.q_tma), nt & 1, abort, lim))) break;
          if (!kSolo && qc == 0) {  // the first query left the exchange slots: the peer may send into them
            mbar_arrive_remote_relaxed(mapa(bar(sh.can_send[0]), peer));
            mbar_arrive_remote_relaxed(mapa(bar(sh.can_send[1]), peer));
          }
          ++qc;
          tc_fence_after();
        }
        const uint32_t b = pc & 1;
        const int st = pc % NS;
        if (pc == (uint32_t)a.stall_page && !(ok = mbar_wait(bar(sh.never), 0, abort, lim))) break;
        if (!(ok = mbar_wait(bar(sh.full[st]), (pc / NS) & 1, abort, lim))) break;
        if (pc >= 2 && !(ok = mbar_wait(bar(sh.s_free[b]), ((pc - 2) >> 1) & 1, abort, lim))) break;
        tc_fence_after();
        const uint32_t sbase = smem_u32(stages + st * kStageBytes);
        const uint64_t kd0 = sdesc_sw128(sbase, 16, 1024);
        const uint64_t kr0 = sdesc_sw64(smem_u32(smem + L::rope_off(st)), 512);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {  // latent: boxes 0..3, 4 K steps each (A = Q in tensor memory)
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ts(tmem + kColS + 64 * b, tmem + kColQ + kk * 8, kd0 + (uint64_t)(off >> 4), idesc_qk_lat,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 2 * L::kRopeBoxes; ++kk)  // RoPE: 32 columns = 2 K steps per box (A = RoPE query tile)
          mma_ss(tmem + kColS + 64 * b, qr0 + (uint64_t)(((kk >> 1) * kQRopeBox + (kk & 1) * 32) >> 4),
                 kr0 + (uint64_t)(((kk >> 1) * kRopeBoxBytes + (kk & 1) * 32) >> 4), idesc_qk, 1u);
        mma_commit(bar(sh.s_full[b]));
        if constexpr (kFp8) mma_commit(bar(sh.rope_empty[st]));
        ++pc;
        c.advance(a);
      }
      if (!ok) fail();
    }
    __syncwarp();  // reconverge before the CTA-wide barrier of the teardown
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P.V issuer
    // Once P.V of page p is done, receive slot p&1 (and the peer's send
    // slot) are free for the peer's next copy: this thread waits for the
    // MMA locally and tells the peer with a relaxed remote arrive (the
    // slot's reads are complete, so no release ordering is needed; a
    // tensor-core commit straight to the peer costs a cluster-scope
    // release, over a thousand cycles on the critical loop).
    if (lane == 0) {
      constexpr uint32_t idesc_pv = kFp8 ? idesc_f16(128, 256, false, true) : idesc_bf16(128, 256, false, true);
      const uint32_t peer_can_send0 = mapa(bar(sh.can_send[0]), peer);
      const uint32_t peer_can_send1 = mapa(bar(sh.can_send[1]), peer);
      PageCursor c;
      c.init(sh.rec, a, lens, lens_raw);
      bool ok = true;
      for (uint32_t p = 0; ok && c.valid; ++p) {
        const uint32_t b = p & 1;
        const bool acc = !c.seg_first();  // a segment's first P.V starts O afresh
        if (!(ok = mbar_wait(bar(sh.p_full[b]), (p >> 1) & 1, abort, lim))) break;
        tc_fence_after();
        const uint64_t pd0 = sdesc_sw128(xrecv + b * kXSlot, 16, 1024);
        const uint64_t vd0 = sdesc_sw128(smem_u32(stages + (p % NS) * kStageBytes), kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 64 tokens = 4 K steps
          mma_ss(tmem + kColO, pd0 + (uint64_t)(kk * 2), vd0 + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                 (acc || kk > 0) ? 1u : 0u);
        mma_commit(bar(sh.empty[p % NS]));
        mma_commit(bar(sh.o_done[b]));
        if constexpr (!kSolo) {
          if (!(ok = mbar_wait(bar(sh.o_done[b]), (p >> 1) & 1, abort, lim))) break;
          mbar_arrive_remote_relaxed(b ? peer_can_send1 : peer_can_send0);
        }
        c.advance(a);
      }
      if (!ok) fail();
    }
    __syncwarp();  // reconverge before the CTA-wide barrier of the teardown
  } else if (warp == R::kIdle) {
    __syncwarp();
  } else if (kFp8 && warp == kDqWarp) {
    // ------------------------------------------------------------ dequantising warp (FP8 cache)
    // Page p: raw slot p % 2 (this CTA's 256 codes of each of the 64 rows,
    // four unswizzled 64 x 64-byte boxes, and the rows' four scales) ->
    // stage p % 3 as f16, c = code value * scale of its 128-column block,
    // in the 128-byte-swizzled K-major layout the TMA gives the bf16 cache.
    // The product is exact for power-of-two scales in [2^-15, 2^7].  Lane j
    // reads 16 codes (a contiguous 512-byte sweep per warp: 8 rows) and
    // writes their 32 bytes to two 16-byte chunks of the row.
    PageCursor c;
    c.init(sh.rec, a, lens, lens_raw);
    bool ok = true;
    for (uint32_t pc = 0; ok && c.valid; ++pc) {
      const int st = pc % NS, rs = pc % kRawSlots;
      ok = mbar_wait(bar(sh.raw_full[rs]), (pc / kRawSlots) & 1, abort, lim);
      if (ok && pc >= (uint32_t)NS) ok = mbar_wait(bar(sh.empty[st]), ((pc / NS) - 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint32_t raw = smem_u32(smem + L::kRawOff + rs * kRawSlotBytes);
      const uint32_t dst = smem_u32(stages + st * kStageBytes);
      // box by box, all eight loads of a box issued before their first use
      // (their shared-memory latencies overlap); the scales of this lane's
      // eight rows, block 2r for boxes 0-1, 2r + 1 for boxes 2-3
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float sc[8];
        uint4 w[8];
        load_scales(raw, 2 * (int)r + (q >> 1), lane, sc);
        load_codes(raw, q, lane, w);
        bad_scale |= dequant_box(w, sc, q, dst, lane);
      }
      fence_proxy_async();  // the stores, seen by the tensor cores' reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(sh.full[st]));
        mbar_arrive(bar(sh.raw_empty[rs]));
      }
      c.advance(a);
    }
    if (!ok && lane == 0) fail();
    __syncwarp();  // reconverge before the CTA-wide barrier of the teardown
  } else if (warp >= kSWarps && warp < kSWarps + kXW) {
    // ------------------------------------------------------------ exchange warps
    // Page p: own partial scores (S_b, fp32) -> 16-bit fixed point with a
    // per-row scale -> send slot b (one row per thread, 128-byte swizzled
    // rows) -> one bulk copy per warp of its 32 rows (4 KiB) and their
    // scales (128 B) into the peer's receive slot b, counted on the peer's
    // barrier of this quadrant.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t peer_recv = mapa(xrecv, peer);
    const uint32_t peer_scale = mapa(smem_u32(&sh.xscale_recv[0][0]), peer);
    const uint32_t peer_xfull0 = mapa(bar(sh.xfull[0][quad]), peer);
    const uint32_t peer_xfull1 = mapa(bar(sh.xfull[1][quad]), peer);
    const int npages = kSolo ? 0 : sh.rec.end - sh.rec.start;  // solo mode: nothing to exchange
    bool ok = true;
    for (int p = 0; ok && p < npages; ++p) {
      const uint32_t b = p & 1;
      ok = mbar_wait(bar(sh.s_full[b]), (p >> 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(lane_base + kColS + 64 * b, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(lane_base + kColS + 64 * b + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(sh.s_free[b]));
      float mx = 0.f;
#pragma unroll
      for (int k = 0; k < 64; k += 2) mx = fmax3(mx, fabsf(__uint_as_float(v[k])), fabsf(__uint_as_float(v[k + 1])));
      const int ke = row_scale_exp(mx);
      const float up = exp2_int(ke);
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 32; ++k)
        w[k] = pack_fixed16x2(__uint_as_float(v[2 * k]) * up, __uint_as_float(v[2 * k + 1]) * up);
      // send slot b is free once our copy of page p-2 has read it
      if (lane == 0 && p >= 2) bulk_wait_read_1();
      __syncwarp();
      const uint32_t dst = xsend + b * kXSlot + row * kXRowBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(dst + ((c ^ (row & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      sh.xscale_send[b][row] = exp2_int(-ke);
      fence_proxy_async();
      // the peer's P.V two pages back (for the first two pages: its first
      // query leaving its slots) freed its receive slot b
      ok = mbar_wait<true>(bar(sh.can_send[b]), (p >> 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        const uint32_t off = b * kXSlot + quad * kXQuadBytes, xb = b ? peer_xfull1 : peer_xfull0;
        const uint32_t soff = (b * kRowsPerCta + quad * 32) * 4;
        bulk_s2s(peer_recv + off, xsend + off, kXQuadBytes, xb);
        bulk_s2s(peer_scale + soff, smem_u32(&sh.xscale_send[0][0]) + soff, kXScaleBytes, xb);
        bulk_commit_group();
      }
      __syncwarp();
      sent = p + 1;
    }
    if (!ok) fail();
  } else {
    // ------------------------------------------------------------ softmax warps
    // Thread = one query row (TMEM lane) and 32 of each page's 64 keys (key
    // half).  Page q: full scores (own S_b in fp32 + the peer's 16-bit
    // partial in receive slot b) -> mask -> row maximum shared with the
    // partner warp -> online softmax -> P (bf16; f16 with an FP8 cache) into receive slot b, over
    // the partial this thread read there, in the layout of an MMA operand.
    // After a failure the loops keep running without work, so every named
    // barrier still sees both warps.
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;  // TMEM lane = query row in this block
    // this CTA's rows: every (l, h) in pair mode; in solo mode (l, h) for
    // the heads h of its latent half, l-major
    const int lrow = (int)rg * kRowsPerCta + row;    // index in this CTA's list
    int l, h, grow;
    bool valid;
    if constexpr (kSolo) {
      const int hh = a.H / 2;                        // heads per l in this CTA's list
      valid = lrow < a.Lq * hh;
      l = valid ? lrow / hh : 0;
      h = valid ? (int)r * hh + lrow % hh : 0;
      grow = l * a.H + h;                            // row of the (l, h) list of all heads
    } else {
      grow = lrow;
      valid = grow < a.rows;
      l = valid ? grow / a.H : 0;
      h = valid ? grow % a.H : 0;
    }
    const int g = (h * a.G) / a.H;
    // The CTA's latent half holds columns 256r .. 256r + 255 of the cache
    // row; this thread fills tensor-memory columns for two 64-column chunks
    // of it (128 * half + 64 * c).  A chunk inside the row's group latent
    // (columns g*d_g .. (g+1)*d_g - 1) takes the query's values from column
    // src_col(c) of its q_cat row; any other chunk is zero, so heads of
    // other groups score nothing against this half.
    // (kept in shared memory: the softmax loop has no registers to spare)
    for (int c = 0; c < 2; ++c) {
      const int col = 256 * (int)r + 128 * half + 64 * c - g * a.d_g;
      sh.qsrc[threadIdx.x][c] = (int16_t)((valid && col >= 0 && col < a.d_g) ? col : -1);
    }
    auto src_col = [&sh](int c) -> int { return sh.qsrc[threadIdx.x][c]; };
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t pair_bar = kBarPair0 + quad;
    const bool leader = (threadIdx.x == 0);
    const int d_q = a.d_g + kDr;
    bool ok = true;

    // this thread's 128 latent query columns of sequence b -> tensor memory;
    // the 128 rows' RoPE half by TMA (rows past the end read as zero; rows
    // of another sequence in a partial block give scores nobody reads)
    auto qrow_of = [&](int b) { return a.q_cat + ((size_t)(b * a.Lq + l) * a.H + h) * d_q; };
    auto load_q = [&](int b) {
      if (!ok) return;
      if (leader) {
        mbar_arrive_expect_tx(bar(sh.q_tma), L::kQRopeBytes);
        if constexpr (kSolo) {
          // all 64 RoPE columns, one run of hh rows (the CTA's heads of one
          // token l) per box; runs past the last token read the next
          // sequence's rows or the zero fill, which nobody uses
          const int hh = a.H / 2;
          for (int run = 0; run < kRowsPerCta / hh; ++run) {
            const int lr = ((int)rg * kRowsPerCta) / hh + run;
            for (int j = 0; j < 2; ++j)
              tma_load_2d(qrope + j * kQRopeBox + run * hh * 64, &tm_qrope, bar(sh.q_tma), a.d_g + 32 * j,
                          (b * a.Lq + lr) * a.H + (int)r * hh);
          }
        } else {
          tma_load_2d(qrope, &tm_qrope, bar(sh.q_tma), a.d_g + 32 * (int)r, b * a.Lq * a.H + (int)rg * kRowsPerCta);
        }
        ++nq_tma;
      }
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // 32 columns (64 bf16) per round trip
        const int sc = src_col(c);
        const uint4* lat = sc >= 0 ? reinterpret_cast<const uint4*>(qrow_of(b) + sc) : nullptr;
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = lat ? lat[k] : make_uint4(0, 0, 0, 0);
          w[4 * k + 0] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
        }
        if constexpr (kFp8) {
          if (query_to_f16(w)) set_status(ws, MLA_ERR_RANGE);
        }
        tmem_st32(lane_base + kColQ + 64 * half + 32 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(sh.q_full));
    };
    // pair mode: pull what this thread will load for sequence b into L2
    // ahead of use (solo mode: the producer warp does it)
    auto prefetch_q = [&](int b) {
      if (!valid) return;
      const char* qrow = reinterpret_cast<const char*>(qrow_of(b));
      const char* lat = qrow + (a.G == 1 ? r * 512 + half * 256 : 0);
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(lat));
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(lat + 128));
      if (half == 0) asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(qrow + a.d_g * 2 + 64 * r));
    };
    auto prefetch_after = [&](const SegIter& at) {  // the sequence after the segment `at` just produced
      SegIter t = at;
      int b2, pa2, pb2;
      if (t.next(a, b2, pa2, pb2)) prefetch_q(b2);
    };

    // the first segment's query: latent half from the exchange slots (box
    // j = 64 columns, 128-byte swizzle), RoPE half already in its tile
    auto load_q_first = [&]() {
      ok = mbar_wait(bar(sh.q_lat), 0, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
        // the box that holds the chunk (the TMA loaded this CTA's half for
        // one group, or the first columns of each row's group latent)
        const int sc = src_col(c);
        const int box = sc < 0 ? 0 : (a.G == 1 ? (sc - 256 * (int)r) / 64 : sc / 64);
        const uint32_t src = xsend + box * kQBoxBytes + row * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          ld_shared_v4(src + ((k ^ (row & 7)) << 4), w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
          if (sc < 0) w[4 * k] = w[4 * k + 1] = w[4 * k + 2] = w[4 * k + 3] = 0u;
        }
        if constexpr (kFp8) {
          if (query_to_f16(w)) set_status(ws, MLA_ERR_RANGE);
        }
        tmem_st32(lane_base + kColQ + 64 * half + 32 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(sh.q_full));
    };

    PageCursor cur;
    cur.init(sh.rec, a, lens, lens_raw);
    if (cur.valid) {
      if constexpr (kSolo) {
        load_q(cur.sb);
      } else {
        load_q_first();
        prefetch_after(cur.it);
      }
    }
    float m_used = -INFINITY, l_part = 0.f;
    int seg = 0, limit = 0;
    uint32_t q = 0;
    while (cur.valid) {
      const uint32_t b = q & 1;
      if (cur.seg_first()) {
        m_used = -INFINITY;
        l_part = 0.f;
        seg = cur.it.slot(cur.sb);
        const int n = cur.it.len(a, cur.sb);
        limit = a.causal ? n - a.Lq + l + 1 : n;  // keys [0, limit) visible
      }
      float s[32];  // raw scores (unscaled) of this thread's 32 keys
      float mt = -INFINITY;
      uint32_t v[32];
      // solo mode: P slot b is free once P.V of page q-2 has read it (in
      // pair mode the peer's copy into the slot already implied that)
      if (kSolo && ok && q >= 2) ok = mbar_wait(bar(sh.o_done[b]), ((q - 2) >> 1) & 1, abort, lim);
      if (ok) ok = mbar_wait(bar(sh.s_full[b]), (q >> 1) & 1, abort, lim);
      if (!kSolo && ok) ok = mbar_wait(bar(sh.xfull[b][quad]), (q >> 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        tmem_ld32(lane_base + kColS + 64 * b + 32 * half, v);  // own scores (partial in pair mode), fp32
        if constexpr (kSolo) {
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(sh.s_free[b]));
#pragma unroll
          for (int k = 0; k < 32; ++k) s[k] = __uint_as_float(v[k]);
        } else {
          const uint32_t src = xrecv + b * kXSlot + row * kXRowBytes;  // the peer's, 16-bit
          uint32_t pw[16];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            ld_shared_v4(src + (((4 * half + c) ^ (row & 7)) << 4), pw[4 * c], pw[4 * c + 1], pw[4 * c + 2],
                         pw[4 * c + 3]);
          const float down = sh.xscale_recv[b][row];
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(sh.s_free[b]));
          // armed for page q+2 (sent by the peer only after our P.V of page q)
          if (half == 0 && lane == 0) mbar_arrive_expect_tx(bar(sh.xfull[b][quad]), kXQuadTx);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 y = unpack_fixed16x2(pw[k]);
            s[2 * k] = fmaf(y.x, down, __uint_as_float(v[2 * k]));
            s[2 * k + 1] = fmaf(y.y, down, __uint_as_float(v[2 * k + 1]));
          }
        }
        const int key0 = cur.i * kPage + 32 * half;
        if (limit < key0 + 32) {  // keys this row may not see
#pragma unroll
          for (int j = 0; j < 32; ++j) s[j] = (key0 + j < limit) ? s[j] : -INFINITY;
        }
        mt = max32(s);
        sh.red[b][half][row] = mt;
      }
      ok = bar_red_and_n(ok, pair_bar, 64);
      if (ok) {
        mt = fmaxf(mt, sh.red[b][half ^ 1][row]) * a.scale_log2;  // log2 units
        const bool need = mt > m_used + kRescaleThreshold;
        if (!cur.seg_first() && __any_sync(0xffffffffu, need)) {  // rescale O once P.V of page q-1 is done
          ok = mbar_wait(bar(sh.o_done[(q - 1) & 1]), ((q - 1) >> 1) & 1, abort, lim);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
            const float f = need ? ex2(m_used - mt) : 1.0f;
            for (int c = 0; c < 8; ++c) {  // 128 columns, 16 at a time
              uint32_t v[16];
              const uint32_t col = lane_base + kColO + 128 * half + 16 * c;
              tmem_ld16(col, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * f);
              tmem_st16(col, v);
            }
            tmem_wait_st();
            tc_fence_before();
            l_part *= f;
          }
        }
        if (ok) {
          if (need) m_used = mt;
          const float base = (m_used == -INFINITY) ? 0.f : m_used;
          uint32_t pk[16];
          float psum = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float p0 = ex2(fmaf(s[2 * j], a.scale_log2, -base));
            const float p1 = ex2(fmaf(s[2 * j + 1], a.scale_log2, -base));
            psum += p0 + p1;  // row sum of the unrounded weights
            pk[j] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
          l_part += psum;
          // P row into receive slot b, over the peer partial this thread
          // read there: K-major, 128-byte swizzle, four 16-byte chunks
          const uint32_t dst = xrecv + b * kXSlot + row * kXRowBytes;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_shared_v4(dst + (((4 * half + c) ^ (row & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                         pk[4 * c + 3]);
          fence_proxy_async();
          mbar_arrive(bar(sh.p_full[b]));
        }
      }
      // every QK of this segment is done (S(q) was complete): the next
      // segment's query, if there is one, may replace it (the cursor copy
      // lives only here, so it costs no registers across the loop)
      if (cur.seg_last()) {
        PageCursor nx = cur;
        nx.advance(a);
        if (nx.valid) {
          load_q(nx.sb);
          if constexpr (!kSolo) prefetch_after(nx.it);
        }
      }

      // ---- end of segment: normalised latent partial and log-sum-exp
      if (cur.seg_last()) {
        if (ok) ok = mbar_wait(bar(sh.o_done[b]), (q >> 1) & 1, abort, lim);  // this page's P.V
        ok = __all_sync(0xffffffffu, ok);
        if (ok) tc_fence_after();
        sh.red[b ^ 1][half][row] = l_part;  // parity of the next page: free until its maximum
        ok = bar_red_and_n(ok, pair_bar, 64);
        const float l_sum = l_part + sh.red[b ^ 1][half ^ 1][row];
        ok = bar_red_and_n(ok, pair_bar, 64);  // both sums read before the next page's maxima land there
        if (ok) {
          const float inv = l_sum > 0.f ? 1.0f / l_sum : 0.f;
          // o_part is chunk-major, [slot][column/4][row][4]: each 16-byte
          // store of a warp covers 512 contiguous bytes (32 consecutive rows).
          float4* dst = reinterpret_cast<float4*>(a.o_part) +
                        ((size_t)seg * (kDc / 4) + r * 64 + half * 32) * a.rows + grow;
          for (int c = 0; c < 8; ++c) {
            uint32_t v[16];
            tmem_ld16(lane_base + kColO + 128 * half + 16 * c, v);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[(size_t)(c * 4 + k) * a.rows] =
                    make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
            }
          }
          if (valid && (kSolo || r == 0) && half == 0)
            a.lse_part[(size_t)seg * a.rows + grow] =
                l_sum > 0.f ? (m_used + lg2(l_sum)) * 0.69314718055994531f : -INFINITY;
          tc_fence_before();
        }
      }
      cur.advance(a);
      ++q;
    }
    if (!ok) fail();
  }

  // ------------------------------------------------------------ teardown
  // Every role has left its loop.  Each thread that started asynchronous
  // work waits (ignoring the abort flag) until it is done: after a normal
  // run these waits return at once; after an abort they keep copies and
  // MMAs from landing in memory that is about to be released.
  // A drain that gives up (nothing in flight should take 100 ms) is
  // recorded as a timeout too, by the thread that gave up.
  if (kFp8 && warp == kDqWarp && __any_sync(0xffffffffu, bad_scale) && lane == 0) set_status(ws, MLA_ERR_RANGE);
  __syncthreads();
  auto drain = [&](uint32_t b, uint32_t parity) {
    if (!mbar_wait_quiet(b, parity)) set_status(a.ws, MLA_ERR_TIMEOUT);
  };
  if (warp == kTmaWarp && lane == 0) {
    if constexpr (kFp8) {  // a page's copies all land on its raw slot's barrier
      for (uint32_t k = issued > (uint32_t)kRawSlots ? issued - kRawSlots : 0; k < issued; ++k)
        drain(bar(sh.raw_full[k % kRawSlots]), (k / kRawSlots) & 1);
    } else {
      for (uint32_t k = issued > (uint32_t)NS ? issued - NS : 0; k < issued; ++k)
        drain(bar(sh.full[k % NS]), (k / NS) & 1);
    }
    if (!kSolo && issued > 0) drain(bar(sh.q_lat), 0);  // the first query's copies
  } else if ((warp == kMmaWarp || warp == kPvWarp) && lane == 0) {
    const int d = warp == kMmaWarp ? 0 : 1;
    mma_commit(bar(sh.drain[d]));
    drain(bar(sh.drain[d]), 0);
  } else if (threadIdx.x == 0 && nq_tma > 0) {
    drain(bar(sh.q_tma), (nq_tma - 1) & 1);
  } else if (warp >= kSWarps && warp < kSWarps + kXW && lane == 0) {
    bulk_wait_read_all();  // this thread's copies have read their send slot
    st_cluster_u32(mapa(smem_u32(&sh.peer_sent[warp - kSWarps]), peer), (uint32_t)sent);
  }
  __syncwarp();
  cluster_sync();  // every copy of the pair issued, the counts of pages sent visible
  // partial scores the peer sent here but this CTA never read (after an
  // abort): its last two pages of each quadrant may still be in flight
  if (warp >= kSWarps && warp < kSWarps + kXW && lane == 0) {
    const int qd = warp - kSWarps, n = sh.peer_sent[qd];
    for (int p = n > 2 ? n - 2 : 0; p < n; ++p) drain(bar(sh.xfull[p & 1][qd]), (p >> 1) & 1);
  }
  __syncwarp();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // neither CTA leaves while the other may still signal it
}
// ---------------------------------------------------------------- plan
// One CTA; used when B is too large for the decode kernel to plan for
// itself.  Validates lengths and table entries, prefix-sums pages per
// sequence and splits the work over `units` clusters with the same rules as
// plan_in_block: two splits are costed in pages (a switch between sequences
// inside a unit counting kSwitchPages) and the cheaper one is written:
//   balanced  — the flattened page list cut into equal contiguous ranges;
//   aligned   — each sequence gets max(1, floor(units * pages_b / total))
//               whole units, at most one per page (needs B <= units), and
//               splits its pages evenly over them.
__global__ void __launch_bounds__(1024)
    plan_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                WsHeader* ws, int B, int Lq, int max_pages, int num_pages, int units) {
  __shared__ int red[33];
  __shared__ int carry, carry2;
  const WsView v = ws_view(ws, B);
  const int tid = threadIdx.x;
  if (tid == 0) carry = carry2 = 0;
  __syncthreads();
  const int lo = Lq > 1 ? Lq : 1, hi = max_pages * kPage;
  for (int base = 0; base < B; base += 1024) {
    const int b = base + tid;
    int np = 0;
    if (b < B) {
      const int n0 = seq_lens[b], n = clamp_len(n0, lo, hi);
      if (n != n0) set_status(ws, MLA_ERR_BAD_SEQLEN);
      v.nlen[b] = n;
      np = (n + kPage - 1) / kPage;
    }
    int sum = 0;
    const int incl = block_scan_incl(np, red, &sum);
    if (b < B) v.off[b] = carry + incl - np;
    __syncthreads();
    if (tid == 0) carry += sum;
    __syncthreads();
  }
  const int total = carry;
  const int chunk = total > 0 ? (total + units - 1) / units : 1;
  if (tid == 0) v.off[B] = total;  // read below by every thread
  __syncthreads();

  int segs = 0;
  for (int k = tid; k < units; k += 1024) {
    const int st = min(k * chunk, total), en = min(st + chunk, total);
    if (st < en) {
      int l0 = 0, h0 = B - 1, l1 = 0, h1 = B - 1;
      while (l0 < h0) { const int m = (l0 + h0 + 1) >> 1; if (v.off[m] <= st) l0 = m; else h0 = m - 1; }
      while (l1 < h1) { const int m = (l1 + h1 + 1) >> 1; if (v.off[m] <= en - 1) l1 = m; else h1 = m - 1; }
      segs = max(segs, l1 - l0 + 1);
    }
  }
  segs = block_reduce_max(segs, red);
  const int cost_bal = chunk + kSwitchPages * (segs - 1);

  int cost_al = INT_MAX, used = 0;
  if (B <= units && total > 0) {
    int worst = 0;
    for (int base = 0; base < B; base += 1024) {
      const int b = base + tid;
      int u = 0;
      if (b < B) {
        const int np = v.off[b + 1] - v.off[b];
        u = aligned_units(np, units, total);
        worst = max(worst, (np + u - 1) / u);
      }
      int sum = 0;
      const int incl = block_scan_incl(u, red, &sum);
      if (b < B) v.slot0[b] = carry2 + incl - u;  // first unit of b (kept if aligned wins)
      __syncthreads();
      if (tid == 0) carry2 += sum;
      __syncthreads();
    }
    used = carry2;
    worst = block_reduce_max(worst, red);
    if (used <= units) cost_al = worst;
  }
  const int mode = cost_al <= cost_bal ? 1 : 0;

  for (int b = tid; b < B; b += 1024) {
    const int o0 = v.off[b], np = v.off[b + 1] - o0;
    if (mode == 1) {
      v.nslot[b] = aligned_units(np, units, total);
    } else {
      const int kf = o0 / chunk, kl = (o0 + np - 1) / chunk;
      v.slot0[b] = b + kf;
      v.nslot[b] = kl - kf + 1;
    }
  }
  __syncthreads();
  for (int k = tid; k < units; k += 1024) {
    UnitRec rec{0, 0, 0, 0, 0};
    if (mode == 1) {
      if (k < used) {
        int l0 = 0, h0 = B - 1;
        while (l0 < h0) { const int m = (l0 + h0 + 1) >> 1; if (v.slot0[m] <= k) l0 = m; else h0 = m - 1; }
        const int nb = v.off[l0 + 1] - v.off[l0], ub = v.nslot[l0], j = k - v.slot0[l0];
        rec = UnitRec{l0, 0, (int)(((long long)j * nb) / ub), (int)(((long long)(j + 1) * nb) / ub), k - l0};
      }
    } else {
      const int st = min(k * chunk, total), en = min(st + chunk, total);
      int l0 = 0, h0 = B - 1;
      while (l0 < h0) { const int m = (l0 + h0 + 1) >> 1; if (v.off[m] <= st) l0 = m; else h0 = m - 1; }
      rec = UnitRec{l0, v.off[l0], st, en, k};
    }
    v.rec[k] = rec;
  }
  if (tid == 0) {
    ws->total = total;
    ws->chunk = chunk;
    ws->units = units;
    ws->B = B;
    ws->mode = mode;
  }
  __syncthreads();
  // table entries actually used must name a real page
  const long long entries = (long long)B * max_pages;
  for (long long e = tid; e < entries; e += 1024) {
    const int b = (int)(e / max_pages), i = (int)(e % max_pages);
    if (i * kPage < v.nlen[b]) {
      const int pg = block_table[e];
      if (pg < 0 || pg >= num_pages) set_status(ws, MLA_ERR_BAD_TABLE);
    }
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* block_table, WsHeader* ws, int B,
                        int Lq, int max_pages, int num_pages, int units, cudaStream_t st) {
  plan_kernel<<<1, 1024, 0, st>>>(seq_lens, block_table, ws, B, Lq, max_pages, num_pages, units);
  return cudaGetLastError();
}

// Per-device facts of the decode launch, found once per device and process
// for each mode of the kernel: whether its shared-memory limit has been
// raised there, and how many clusters of 2, 4, 6 and 8 CTAs fit at once.
// Calls may come from several host threads and for several devices, so the
// table is guarded by a mutex (never held across a CUDA call).  Devices past
// the table are not cached.
namespace {
constexpr int kCachedDevices = 64;
struct DecodeDeviceInfo {
  bool smem_set[2][2];  // [solo][fp8]
  int units[2][2][4];   // [solo][fp8][clusters of 2, 4, 6, 8 CTAs]; 0 = not known yet
};
std::mutex g_decode_mu;
DecodeDeviceInfo g_decode_info[kCachedDevices];

template <bool kSolo, bool kFp8>
cudaError_t decode_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int units, int csize,
                          cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kCachedDevices;
  bool set = false;
  if (cached) {
    std::lock_guard<std::mutex> lock(g_decode_mu);
    set = g_decode_info[dev].smem_set[kSolo][kFp8];
  }
  if (!set) {  // the attribute is per device
    e = cudaFuncSetAttribute(decode_kernel<kSolo, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             decode_smem<kSolo, kFp8>());
    if (e != cudaSuccess) return e;
    if (cached) {
      std::lock_guard<std::mutex> lock(g_decode_mu);
      g_decode_info[dev].smem_set[kSolo][kFp8] = true;
    }
  }
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(units * csize);
  cfg.blockDim = dim3(Roles<kSolo, kFp8>::kThreads);
  cfg.dynamicSmemBytes = decode_smem<kSolo, kFp8>();
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaSuccess;
}

template <bool kSolo, bool kFp8>
int decode_max_units_mode(int csize, int* units) {
  const int slot = csize / 2 - 1;
  if (slot < 0 || slot > 3 || (csize & 1)) return MLA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  const bool cached = dev >= 0 && dev < kCachedDevices;
  if (cached) {
    std::lock_guard<std::mutex> lock(g_decode_mu);
    if (g_decode_info[dev].units[kSolo][kFp8][slot] > 0) {
      *units = g_decode_info[dev].units[kSolo][kFp8][slot];
      return MLA_OK;
    }
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  if (decode_config<kSolo, kFp8>(cfg, attr, 1, csize, nullptr) != cudaSuccess) return MLA_ERR_CUDA;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<kSolo, kFp8>, &cfg) != cudaSuccess || n < 1)
    return MLA_ERR_CUDA;
  if (n > kMaxUnits) n = kMaxUnits;  // the workspace holds per-unit records for at most this many
  if (cached) {
    std::lock_guard<std::mutex> lock(g_decode_mu);
    g_decode_info[dev].units[kSolo][kFp8][slot] = n;
  }
  *units = n;
  return MLA_OK;
}
}  // namespace

int decode_max_units(bool solo, bool fp8, int csize, int* units) {
  if (fp8) return solo ? decode_max_units_mode<true, true>(csize, units) : decode_max_units_mode<false, true>(csize, units);
  return solo ? decode_max_units_mode<true, false>(csize, units) : decode_max_units_mode<false, false>(csize, units);
}

namespace {
template <bool kSolo, bool kFp8>
cudaError_t launch_decode_mode(const CUtensorMap& tm_cache, const CUtensorMap& tm_rope, const CUtensorMap& tm_qrope,
                               const CUtensorMap& tm_qlat, const CUtensorMap& tm_scale, const DecodeArgs& a,
                               int units, int csize, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cudaError_t e = decode_config<kSolo, kFp8>(cfg, attr, units, csize, st);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_kernel<kSolo, kFp8>, tm_cache, tm_rope, tm_qrope, tm_qlat, tm_scale, a);
}
}  // namespace

cudaError_t launch_decode(bool solo, bool fp8, const CUtensorMap& tm_cache, const CUtensorMap& tm_rope,
                          const CUtensorMap& tm_qrope, const CUtensorMap& tm_qlat, const CUtensorMap& tm_scale,
                          const DecodeArgs& a, int units, int csize, cudaStream_t st) {
  if (fp8)
    return solo ? launch_decode_mode<true, true>(tm_cache, tm_rope, tm_qrope, tm_qlat, tm_scale, a, units, csize, st)
                : launch_decode_mode<false, true>(tm_cache, tm_rope, tm_qrope, tm_qlat, tm_scale, a, units, csize, st);
  return solo ? launch_decode_mode<true, false>(tm_cache, tm_rope, tm_qrope, tm_qlat, tm_scale, a, units, csize, st)
              : launch_decode_mode<false, false>(tm_cache, tm_rope, tm_qrope, tm_qlat, tm_scale, a, units, csize, st);
}

}  // namespace mla
