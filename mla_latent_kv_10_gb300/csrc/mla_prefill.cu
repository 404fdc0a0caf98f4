// mla_prefill.cu — the decompress branch for long query chunks: the latent
// cache is expanded into per-head keys and values, then dense causal
// attention runs over them (MLA operator write-up §3: the plugin's prefill
// threshold of 256 query tokens; §6: long chunks take the decompressing
// path, short ones the absorbed one).
//
//   decompress: k_nope[b,h,s,:] = W_UK[h] . c_g(h)[s]      (128 values)
//               v[b,h,s,:]      = W_UV[h] . c_g(h)[s]      (128 values)
//               for every cached token s < n_b, zeros for s in [n_b, 64 *
//               pages(n_b)) so that no masked key can carry a non-finite
//               value into P.V.  Layout [B, H, S, 128] bf16, S =
//               max_pages_per_seq * 64.
//   attend:     out[b,l,h,:] = softmax_s((q_nope . k_nope[s] + q_rope .
//               k_R[s]) * scale) . v[s], keys s <= n_b - Lq + l (causal,
//               the new tokens last), lse[b,l,h] the natural log-sum-exp.
//               k_R[s] is read from the cache rows (columns 512..575).
//
// GB300 design: tcgen05 MMAs with fp32 accumulators in tensor memory,
// operands staged by TMA with 128-byte swizzle, mbarrier pipelines with
// bounded waits (a wait that gives up records MLA_ERR_TIMEOUT, the CTA
// drains what it started and returns).
#include <cmath>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void set_status(WsHeader* ws, int code) { atomicCAS(&ws->status, 0, code); }

// sequence length of b, clamped into [lo, hi] (a change is reported)
__device__ __forceinline__ int seq_len_checked(const int32_t* seq_lens, int b, int lo, int hi, WsHeader* ws,
                                               bool report) {
  const int n0 = seq_lens[b];
  const int n = n0 < lo ? lo : (n0 > hi ? hi : n0);
  if (report && n != n0) set_status(ws, MLA_ERR_BAD_SEQLEN);
  return n;
}

// page id i of sequence b, replaced by page 0 (and reported) when out of range
__device__ __forceinline__ int page_checked(const int32_t* block_table, int b, int i, int max_pages,
                                            int num_pages, WsHeader* ws) {
  int p = block_table[(size_t)b * max_pages + i];
  if (p < 0 || p >= num_pages) {
    set_status(ws, MLA_ERR_BAD_TABLE);
    p = 0;
  }
  return p;
}

// 32 fp32 accumulator columns of one row -> bf16 (64 bytes)
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32], float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * mul, __uint_as_float(r[8 * q + 1]) * mul);
    v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * mul, __uint_as_float(r[8 * q + 3]) * mul);
    v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * mul, __uint_as_float(r[8 * q + 5]) * mul);
    v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * mul, __uint_as_float(r[8 * q + 7]) * mul);
    d[q] = v;
  }
}

constexpr int kTile = 64 * 64 * 2;  // a 64-row x 64-column bf16 box, 128-byte swizzle: 8 KiB

// ---------------------------------------------------------------- decompress
// One CTA per (head h, two pages of sequence b): M = 128 tokens, N = 128
// output values, K = d_g latent columns streamed in 64-column chunks
// through a 2-slot ring.  A slot holds the two pages' rows of the chunk
// (two 64-row boxes, 16 KiB) and the chunk of W_UK[h] and of W_UV[h]
// (128 x 64 each, K-major, 16 KiB each).  D_K in tensor-memory columns
// 0..127, D_V in 128..255.  Thread 0 issues copies and MMAs; the four warps
// (tensor-memory lane = token) store the rows.  Two slots (96 KiB) let two
// CTAs share an SM, so one's copies overlap the other's MMAs and stores
// (three slots, one CTA per SM, measured 35 % slower).
constexpr int kDcSlots = 2, kDcSlot = 2 * kTile + 2 * 2 * kTile;  // 48 KiB
constexpr int kDcSmem = kDcSlots * kDcSlot + 1024;
template <int DG>
__global__ void __launch_bounds__(128)
    decompress_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmWK,
                      const __grid_constant__ CUtensorMap tmWV, const int32_t* __restrict__ block_table,
                      const int32_t* __restrict__ seq_lens, __nv_bfloat16* __restrict__ k_nope,
                      __nv_bfloat16* __restrict__ v_out, WsHeader* ws, int H, int G, int Lq, int max_pages,
                      int num_pages, unsigned long long wait_ns) {
  constexpr int kChunks = DG / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(8) uint64_t bars[2 * kDcSlots + 2];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  const int h = blockIdx.x, t = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = max_pages * kPage;
  griddep_wait();
  const int n = seq_len_checked(seq_lens, b, Lq, S, ws, threadIdx.x == 0 && h == 0 && t == 0);
  const int npages = (n + kPage - 1) / kPage;
  if (2 * t >= npages) return;  // the whole block leaves before any set-up
  const int g = (h * G) / H;
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kDcSlots + s]); };
  const uint32_t done = smem_u32(&bars[2 * kDcSlots]), drain = smem_u32(&bars[2 * kDcSlots + 1]);
  auto slotA = [&](int s) { return smem_u32(smem + s * kDcSlot); };
  auto slotK = [&](int s) { return smem_u32(smem + s * kDcSlot + 2 * kTile); };
  auto slotV = [&](int s) { return smem_u32(smem + s * kDcSlot + 4 * kTile); };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kDcSlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmWK);
    tma_prefetch_desc(&tmWV);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;

  int issued = 0;  // thread 0: chunks whose copies were issued
  if (threadIdx.x == 0) {
    const int pg0 = page_checked(block_table, b, 2 * t, max_pages, num_pages, ws);
    const int pg1 = 2 * t + 1 < npages ? page_checked(block_table, b, 2 * t + 1, max_pages, num_pages, ws) : pg0;
    auto load = [&](int c) {
      const int s = c % kDcSlots, col = g * DG + 64 * c;
      mbar_arrive_expect_tx(full(s), kDcSlot);
      tma_load_2d(slotA(s), &tmC, full(s), col, pg0 * kPage);
      tma_load_2d(slotA(s) + kTile, &tmC, full(s), col, pg1 * kPage);
      tma_load_3d(slotK(s), &tmWK, full(s), 64 * c, 0, h);
      tma_load_3d(slotV(s), &tmWV, full(s), 64 * c, 0, h);
      ++issued;
    };
    for (int c = 0; c < kChunks && c < kDcSlots; ++c) load(c);
    constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
    bool ok = true;
    for (int c = 0; c < kChunks && ok; ++c) {
      const int s = c % kDcSlots;
      if (!(ok = mbar_wait(full(s), (c / kDcSlots) & 1, &abort_flag, wait_ns))) break;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // K = 64 in steps of 16
        const uint64_t ad = sdesc_sw128(slotA(s) + j * 32, 16, 1024);
        const uint32_t acc = (c > 0 || j > 0) ? 1u : 0u;
        mma_ss(tmem, ad, sdesc_sw128(slotK(s) + j * 32, 16, 1024), idesc, acc);
        mma_ss(tmem + 128, ad, sdesc_sw128(slotV(s) + j * 32, 16, 1024), idesc, acc);
      }
      mma_commit(empty(s));
      if (c + kDcSlots < kChunks) {
        if (!(ok = mbar_wait(empty(s), (c / kDcSlots) & 1, &abort_flag, wait_ns))) break;
        load(c + kDcSlots);
      }
    }
    if (ok) {
      mma_commit(done);
    } else {
      abort_flag = 1;
      set_status(ws, MLA_ERR_TIMEOUT);
    }
  }
  __syncwarp();  // warp 0 reconverges before the aligned tensor-memory loads below
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, &abort_flag, wait_ns));
  tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane, s = 128 * t + row;  // token of this thread
    if (s < npages * kPage) {
      const size_t o = (((size_t)b * H + h) * S + s) * kDhc;
      const float keep = s < n ? 1.0f : 0.0f;  // rows past the sequence's end: zeros
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {  // 4 x 32 columns of K, then of V
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k)  // 0 * NaN would stay NaN: replace, do not scale
          if (keep == 0.0f) r[k] = 0u;
        store32_bf16((c < 4 ? k_nope : v_out) + o + (c & 3) * 32, r, 1.0f);
      }
    }
  }
  // teardown: copies and MMAs still in flight land before the memory goes
  if (threadIdx.x == 0) {
    for (int c = issued > kDcSlots ? issued - kDcSlots : 0; c < issued; ++c)
      if (!mbar_wait_quiet(full(c % kDcSlots), (c / kDcSlots) & 1)) set_status(ws, MLA_ERR_TIMEOUT);
    mma_commit(drain);
    if (!mbar_wait_quiet(drain, 0)) set_status(ws, MLA_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------- attend
// One CTA per (128 query rows of head h of sequence b), 224 threads:
//   warps 0-3  softmax: thread = query row = tensor-memory lane; the whole
//              row's 64 keys of a page, online softmax in fp32 (O is
//              rescaled only when the row maximum has grown by 2^8),
//              P (bf16) into its slot as the A operand of P.V, epilogue;
//   warp 4     TMA producer (lane 0): the query tile once, then per page
//              the 64 keys' k_nope (two boxes), k_R (from the cache row)
//              and v (two boxes) into a 3-stage ring;
//   warps 5, 6 the QK and the P.V issuers (lane 0 each): S(p+1) = Q . K^T
//              waits only for its page and score buffer, so the tensor pipe
//              works while the softmax does.  (One thread issuing both,
//              QK(p+2) queued behind P(p) . V, measured slower; two softmax
//              threads per row, 32 keys each, measured 4 % slower.)
// Tensor memory: O (128 columns) | S0, S1 (64 each).
constexpr int kAtStages = 3;
constexpr int kAtQ = 3 * 2 * kTile;              // 128 rows x 192 columns: three 128 x 64 boxes, 48 KiB
constexpr int kAtStage = 3 * kTile + 2 * kTile;  // K: nope (2 boxes) + RoPE (1 box); V: 2 boxes; 40 KiB
constexpr int kAtP = 2 * kTile;                  // 128 rows x 64 keys bf16, 16 KiB
constexpr int kAtSmem = kAtQ + kAtStages * kAtStage + 2 * kAtP + 1024;
constexpr float kAtRescale = 8.0f;  // log2 units

struct AtArgs {
  const int32_t* block_table;
  const int32_t* seq_lens;
  __nv_bfloat16* out;
  float* lse;
  WsHeader* ws;
  int B, Lq, H, S, max_pages, num_pages;
  float scale_log2;
  unsigned long long wait_ns;
};

__device__ __forceinline__ float at_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(224, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmQN, const __grid_constant__ CUtensorMap tmQR,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmC, const AtArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sQ = smem_u32(smem);
  auto sK = [&](int st) { return smem_u32(smem + kAtQ + st * kAtStage); };
  auto sV = [&](int st) { return smem_u32(smem + kAtQ + st * kAtStage + 3 * kTile); };
  auto sP = [&](int b) { return smem_u32(smem + kAtQ + kAtStages * kAtStage + b * kAtP); };
  __shared__ __align__(8) uint64_t full[kAtStages], empty[kAtStages], q_full, s_full[2], s_free[2], p_full[2],
      o_done[2], drain;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  auto bar = [](uint64_t& x) { return smem_u32(&x); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int l0 = blockIdx.x * kRowsPerCta, h = blockIdx.y, b = blockIdx.z;
  const unsigned long long lim = a.wait_ns;
  griddep_wait();
  const int n = seq_len_checked(a.seq_lens, b, a.Lq, a.S, a.ws, threadIdx.x == 0 && h == 0 && blockIdx.x == 0);
  const int l_last = min(l0 + kRowsPerCta, a.Lq) - 1;
  const int npg = (n - a.Lq + l_last) / kPage + 1;  // pages holding keys some row of the block sees
  const int kv_row0 = (b * a.H + h) * a.S;          // row of key 0 in the [B*H*S, 128] views

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(bar(full[s]), 1);
      mbar_init(bar(empty[s]), 2);  // the K half (QK done) and the V half (P.V done)
    }
    mbar_init(bar(q_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(s_full[s]), 1);
      mbar_init(bar(s_free[s]), 128);
      mbar_init(bar(p_full[s]), 128);
      mbar_init(bar(o_done[s]), 1);
    }
    mbar_init(bar(drain), 2);
    fence_mbar_init();
    tma_prefetch_desc(&tmQN);
    tma_prefetch_desc(&tmQR);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&tmem_holder), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  volatile int* abort = &abort_flag;
  auto fail = [&]() {
    *abort = 1;
    set_status(a.ws, MLA_ERR_TIMEOUT);
  };
  int issued = 0;  // producer: pages whose copies were issued

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int qrow = b * a.Lq + l0;
      mbar_arrive_expect_tx(bar(q_full), kAtQ);
      tma_load_2d(sQ, &tmQN, bar(q_full), h * kDhc, qrow);
      tma_load_2d(sQ + 2 * kTile, &tmQN, bar(q_full), h * kDhc + 64, qrow);
      tma_load_2d(sQ + 4 * kTile, &tmQR, bar(q_full), h * kDr, qrow);
      bool ok = true;
      for (int p = 0; p < npg; ++p) {
        const int st = p % kAtStages;
        if (p >= kAtStages && !(ok = mbar_wait(bar(empty[st]), ((p / kAtStages) - 1) & 1, abort, lim))) break;
        const int page = page_checked(a.block_table, b, p, a.max_pages, a.num_pages, a.ws);
        mbar_arrive_expect_tx(bar(full[st]), kAtStage);
        tma_load_2d(sK(st), &tmK, bar(full[st]), 0, kv_row0 + p * kPage);
        tma_load_2d(sK(st) + kTile, &tmK, bar(full[st]), 64, kv_row0 + p * kPage);
        tma_load_2d(sK(st) + 2 * kTile, &tmC, bar(full[st]), kDc, page * kPage);
        tma_load_2d(sV(st), &tmV, bar(full[st]), 0, kv_row0 + p * kPage);
        tma_load_2d(sV(st) + kTile, &tmV, bar(full[st]), 64, kv_row0 + p * kPage);
        ++issued;
      }
      if (!ok) fail();
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ QK issuer
    // S(p & 1) = Q . K(p)^T once page p landed and the softmax has read
    // S(p - 2); the stage's K half is free once these MMAs are done.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, 64, false, false);
      bool ok = mbar_wait(bar(q_full), 0, abort, lim);
      for (int p = 0; ok && p < npg; ++p) {
        const int st = p % kAtStages;
        if (!(ok = mbar_wait(bar(full[st]), (p / kAtStages) & 1, abort, lim))) break;
        if (p >= 2 && !(ok = mbar_wait(bar(s_free[p & 1]), ((p - 2) >> 1) & 1, abort, lim))) break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 12; ++j) {  // 12 K steps of 16 over 192 columns
          const uint64_t ad = sdesc_sw128(sQ + (j >> 2) * 2 * kTile + (j & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sK(st) + (j >> 2) * kTile + (j & 3) * 32, 16, 1024);
          mma_ss(tmem + 128 + 64 * (p & 1), ad, bd, idesc_qk, j > 0 ? 1u : 0u);
        }
        mma_commit(bar(s_full[p & 1]));
        mma_commit(bar(empty[st]));
      }
      if (!ok) fail();
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ P.V issuer
    // O += P(p) . V(p) once the softmax has written P(p); the stage's V half
    // and P slot p & 1 are free once these MMAs are done.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
      bool ok = true;
      for (int p = 0; ok && p < npg; ++p) {
        if (!(ok = mbar_wait(bar(p_full[p & 1]), (p >> 1) & 1, abort, lim))) break;
        tc_fence_after();
        const int st = p % kAtStages;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 64 keys = 4 K steps
          const uint64_t ad = sdesc_sw128(sP(p & 1) + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sV(st) + kk * 2048, kTile, 1024);
          mma_ss(tmem, ad, bd, idesc_pv, (p > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(empty[st]));
        mma_commit(bar(o_done[p & 1]));
      }
      if (!ok) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = warp * 32 + lane, l = l0 + row;
    const bool valid = l < a.Lq;
    const int vis = valid ? n - a.Lq + l + 1 : 0;  // keys [0, vis) visible to this row
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int p = 0; p < npg; ++p) {
      const int sb = p & 1;
      float s[64];
      if (ok) ok = mbar_wait(bar(s_full[sb]), (p >> 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(lane_base + 128 + 64 * sb, v0);
        tmem_ld32(lane_base + 128 + 64 * sb + 32, v1);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          s[k] = __uint_as_float(v0[k]);
          s[32 + k] = __uint_as_float(v1[k]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(s_free[sb]));
      const int key0 = p * kPage;
      if (vis < key0 + kPage) {
#pragma unroll
        for (int k = 0; k < 64; ++k) s[k] = key0 + k < vis ? s[k] : -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int k = 1; k < 64; ++k) mx = fmaxf(mx, s[k]);
      mx *= a.scale_log2;
      const bool need = mx > m_used + kAtRescale;
      if (p > 0 && __any_sync(0xffffffffu, need)) {  // rescale O once P.V of page p-1 is done
        ok = mbar_wait(bar(o_done[(p - 1) & 1]), ((p - 1) >> 1) & 1, abort, lim);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float f = need ? at_ex2(m_used - mx) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[16];
          tmem_ld16(lane_base + 16 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * f);
          tmem_st16(lane_base + 16 * c, v);
        }
        tmem_wait_st();
        tc_fence_before();
        l_sum *= f;
      }
      if (need) m_used = mx;
      const float base = m_used == -INFINITY ? 0.f : m_used;
      // P slot sb is free once P.V of page p-2 has read it
      if (p >= 2) ok = mbar_wait(bar(o_done[sb]), ((p - 2) >> 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p0 = at_ex2(fmaf(s[2 * j], a.scale_log2, -base));
        const float p1 = at_ex2(fmaf(s[2 * j + 1], a.scale_log2, -base));
        psum += p0 + p1;
        pk[j] = pack_bf16x2(p0, p1);
      }
      l_sum += psum;
      // row of P: 64 keys = 128 bytes, K-major with 128-byte swizzle
      const uint32_t dst = sP(sb) + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + ((c ^ (row & 7)) << 4)),
                     "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(bar(p_full[sb]));
    }
    // epilogue: O / l -> out (bf16), lse
    if (ok) ok = mbar_wait(bar(o_done[(npg - 1) & 1]), ((npg - 1) >> 1) & 1, abort, lim);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const float inv = l_sum > 0.f ? 1.0f / l_sum : 0.f;
      __nv_bfloat16* dst = a.out + (((size_t)b * a.Lq + (valid ? l : 0)) * a.H + h) * kDhc;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + 32 * c, r);
        tmem_wait_ld();
        if (valid) store32_bf16(dst + 32 * c, r, inv);
      }
      if (valid)
        a.lse[((size_t)b * a.Lq + l) * a.H + h] =
            l_sum > 0.f ? (m_used + __log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
    } else {
      fail();
    }
  }

  // teardown: copies and MMAs still in flight land before the memory goes
  __syncthreads();
  if (warp == 4 && lane == 0) {
    for (int p = issued > kAtStages ? issued - kAtStages : 0; p < issued; ++p)
      if (!mbar_wait_quiet(bar(full[p % kAtStages]), (p / kAtStages) & 1)) set_status(a.ws, MLA_ERR_TIMEOUT);
    if (!mbar_wait_quiet(bar(q_full), 0)) set_status(a.ws, MLA_ERR_TIMEOUT);
  } else if ((warp == 5 || warp == 6) && lane == 0) {  // each issuer's MMAs done
    mma_commit(bar(drain));
    if (!mbar_wait_quiet(bar(drain), 0)) set_status(a.ws, MLA_ERR_TIMEOUT);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

template <int DG>
cudaError_t launch_decompress_dg(const CUtensorMap& tmC, const CUtensorMap& tmWK, const CUtensorMap& tmWV,
                                 const int32_t* block_table, const int32_t* seq_lens, void* k_nope, void* v,
                                 WsHeader* ws, int B, int H, int G, int Lq, int max_pages, int num_pages,
                                 unsigned long long wait_ns, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(decompress_kernel<DG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDcSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(H, (max_pages + 1) / 2, B), block(128);
  decompress_kernel<DG><<<grid, block, kDcSmem, st>>>(tmC, tmWK, tmWV, block_table, seq_lens,
                                                      static_cast<__nv_bfloat16*>(k_nope),
                                                      static_cast<__nv_bfloat16*>(v), ws, H, G, Lq, max_pages,
                                                      num_pages, wait_ns);
  return cudaGetLastError();
}

cudaError_t launch_decompress(const CUtensorMap& tmC, const CUtensorMap& tmWK, const CUtensorMap& tmWV,
                              const int32_t* block_table, const int32_t* seq_lens, void* k_nope, void* v,
                              WsHeader* ws, int B, int H, int G, int Lq, int max_pages, int num_pages,
                              unsigned long long wait_ns, cudaStream_t st) {
  switch (kDc / G) {
    case 512: return launch_decompress_dg<512>(tmC, tmWK, tmWV, block_table, seq_lens, k_nope, v, ws, B, H, G, Lq,
                                               max_pages, num_pages, wait_ns, st);
    case 256: return launch_decompress_dg<256>(tmC, tmWK, tmWV, block_table, seq_lens, k_nope, v, ws, B, H, G, Lq,
                                               max_pages, num_pages, wait_ns, st);
    case 128: return launch_decompress_dg<128>(tmC, tmWK, tmWV, block_table, seq_lens, k_nope, v, ws, B, H, G, Lq,
                                               max_pages, num_pages, wait_ns, st);
    case 64: return launch_decompress_dg<64>(tmC, tmWK, tmWV, block_table, seq_lens, k_nope, v, ws, B, H, G, Lq,
                                             max_pages, num_pages, wait_ns, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill_attend(const CUtensorMap& tmQN, const CUtensorMap& tmQR, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, const CUtensorMap& tmC, const int32_t* block_table,
                                  const int32_t* seq_lens, void* out, float* lse, WsHeader* ws, int B, int Lq,
                                  int H, int max_pages, int num_pages, float scale, unsigned long long wait_ns,
                                  cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAtSmem);
  if (e != cudaSuccess) return e;
  AtArgs a;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.ws = ws;
  a.B = B;
  a.Lq = Lq;
  a.H = H;
  a.S = max_pages * kPage;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = wait_ns;
  dim3 grid((Lq + kRowsPerCta - 1) / kRowsPerCta, H, B), block(224);
  prefill_attn_kernel<<<grid, block, kAtSmem, st>>>(tmQN, tmQR, tmK, tmV, tmC, a);
  return cudaGetLastError();
}

}  // namespace mla
