// mla_combine.cu — log-sum-exp merge of the split-KV partials written by the
// decode kernel: alone (combine_kernel: latent output o_lat in bf16 and the
// row log-sum-exp), or inside the W_UV projection (combine_project_kernel:
// the merged latent rows go straight into shared memory as the A operand of
// the tensor-core product out = o_lat . W_UV[h]^T).
//
// The MLA pages name split-KV decoding but give no merge; this is the exact
// identity of a softmax taken over disjoint key ranges.  A split s of a query
// row holds o_s = (sum_k p_k v_k) / l_s and lse_s = m_s + log l_s over its
// keys; the row's result is L = log sum_s exp(lse_s) and
// o = sum_s exp(lse_s - L) o_s.  Splits with no keys carry lse = -inf and
// weigh nothing.  The partials are fp32 chunk-major, [slot][column/4][row][4]
// (row = l*H + h); sequence b owns slots slot0[b] .. slot0[b] + nslot[b] - 1
// of the workspace.  A plan written for another
// batch is not followed, and every slot range is clipped to the `slots`
// partials the caller allocated.
#include <atomic>
#include <cmath>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// One row merged by a warp: slot range [s0, s0 + nseg); lane i sums the K
// 8-column chunks ch[k] (two float4 chunks each of the chunk-major
// partials).  The first kBatch partials are requested
// together with the row's log-sum-exps, so the row costs one memory round
// trip when it has at most kBatch partials.  L receives the row's
// log-sum-exp.
template <int K>
__device__ __forceinline__ void merge_row(int s0, int nseg, const float* __restrict__ o_part,
                                          const float* __restrict__ lse_part, int row, int rows,
                                          const int (&ch)[K], float4 (&acc)[K][2], float& L) {
  constexpr int kBatch = 2;
  const int lane = threadIdx.x & 31;
  const float4* base = reinterpret_cast<const float4*>(o_part) + row;
  const size_t slot_stride = (size_t)(kDc / 4) * rows;
#pragma unroll
  for (int k = 0; k < K; ++k) acc[k][0] = acc[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 pv[kBatch][K][2];
  auto issue = [&](int j0) {
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj) {
      const float4* src = base + (size_t)(s0 + j0 + jj) * slot_stride;
#pragma unroll
      for (int k = 0; k < K; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          pv[jj][k][e] = j0 + jj < nseg ? __ldcg(src + (size_t)(2 * ch[k] + e) * rows) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  issue(0);
  const float x0 = lane < nseg ? lse_part[(size_t)(s0 + lane) * rows + row] : -INFINITY;
  const float x1 = lane + 32 < nseg ? lse_part[(size_t)(s0 + lane + 32) * rows + row] : -INFINITY;
  float mx = fmaxf(x0, x1);
  for (int j = lane + 64; j < nseg; j += 32) mx = fmaxf(mx, lse_part[(size_t)(s0 + j) * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  if (mx != -INFINITY) {
    sum = expf(x0 - mx) + expf(x1 - mx);
    for (int j = lane + 64; j < nseg; j += 32) sum += expf(lse_part[(size_t)(s0 + j) * rows + row] - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  L = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
  const float w0 = L == -INFINITY ? 0.f : expf(x0 - L), w1 = L == -INFINITY ? 0.f : expf(x1 - L);
#pragma unroll 1
  for (int j0 = 0; j0 < nseg; j0 += kBatch) {
    if (j0 > 0) issue(j0);
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj) {
      const int j = j0 + jj;
      float w = 0.f;
      if (j < nseg) {  // warp-uniform
        if (j < 32) w = __shfl_sync(0xffffffffu, w0, j);
        else if (j < 64) w = __shfl_sync(0xffffffffu, w1, j - 32);
        else w = L == -INFINITY ? 0.f : expf(lse_part[(size_t)(s0 + j) * rows + row] - L);
      }
#pragma unroll
      for (int k = 0; k < K; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          acc[k][e].x = fmaf(w, pv[jj][k][e].x, acc[k][e].x);
          acc[k][e].y = fmaf(w, pv[jj][k][e].y, acc[k][e].y);
          acc[k][e].z = fmaf(w, pv[jj][k][e].z, acc[k][e].z);
          acc[k][e].w = fmaf(w, pv[jj][k][e].w, acc[k][e].w);
        }
    }
  }
}

// ---------------------------------------------------------------- combine
// One CTA of 512 threads per (sequence, 32 query rows, 256 latent columns):
// one CTA fits an SM at a time, so a grid of about one CTA per SM finishes
// in one wave.  The first partials' loads are issued before the row
// weights are known, so the CTA waits for two dependent global round trips
// (the plan's batch with the sequence's split record, then log-sum-exps and
// partials together), not three.
// The log-sum-exp of each row's partials is reduced with warp shuffles over
// the partial index and turned into per-partial weights in shared memory;
// the weighted sum reads the chunk-major partials coalesced (32 consecutive
// rows per warp access).  The bf16 result is staged in shared memory and
// written out as contiguous row pieces.
// A grid of more CTAs than SMs (many sequences, or several query rows a
// sequence) runs the 256-thread form instead: each thread sums twice the
// chunks with half the partials in flight, and two CTAs share an SM, so
// one CTA's round trips overlap the other's.
constexpr int kCombineRows = 32, kCombineCols = 256, kCombineMaxSeg = 64, kCombineThreads = 512;
template <int DG, int kThreads, int kBatch>
__global__ void __launch_bounds__(kThreads, kCombineThreads / kThreads)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                   const WsHeader* __restrict__ ws, __nv_bfloat16* __restrict__ o_lat,
                   float* __restrict__ lse_out, int B, int Lq, int H, int G, int slots) {
  constexpr int kCols = DG < kCombineCols ? DG : kCombineCols;  // columns of this CTA
  constexpr int kWarps = kThreads / 32;
  static_assert(DG % kCols == 0 && (kCols / 4) % kWarps == 0, "latent slice in whole CTA column ranges");
  __shared__ __align__(16) __nv_bfloat16 tile[kCombineRows][kCols + 8];
  __shared__ float wts[kCombineMaxSeg][kCombineRows];
  __shared__ float lrow[kCombineRows];
  const int rows = Lq * H;
  const int b = blockIdx.x, r0 = blockIdx.y * kCombineRows, cz = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  // the plan's batch and this sequence's split record are requested
  // together (their places follow from the argument B, and the workspace
  // holds at least that much); a plan written for another batch is not
  // followed
  const WsView v = ws_view(ws, B);
  const int plan_b = ws->B, s0r = v.slot0[b], nsl = v.nslot[b];
  if (plan_b != B) return;
  const int nseg = (s0r < 0 || s0r >= slots) ? 0 : min(nsl, slots - s0r);
  const size_t seg0 = (size_t)(s0r < 0 ? 0 : s0r);
  const bool table = nseg <= kCombineMaxSeg;

  // weighted-sum thread layout: (row lane, chunk group warp); the first
  // kBatch partials of the thread's chunks are requested right away
  const int row = r0 + lane;
  const bool valid = row < rows;
  const int h = valid ? row % H : 0, g = (h * G) / H;
  constexpr int kChunks = kCols / 4, kPer = kChunks / kWarps;  // chunks of this thread: warp + kWarps*k
  // kBatch: partials whose loads are all issued before any is used
  const float4* src = reinterpret_cast<const float4*>(o_part) +
                      (size_t)(g * (DG / 4) + cz * kChunks + warp) * rows + row;
  const size_t slot_stride = (size_t)(kDc / 4) * rows, chunk_stride = (size_t)kWarps * rows;
  float4 pv[kBatch][kPer];
  auto issue = [&](int j0) {
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj) {
      const float4* sj = src + (seg0 + j0 + jj) * slot_stride;
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        pv[jj][k] = (valid && j0 + jj < nseg) ? __ldcs(sj + k * chunk_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };

  // log-sum-exp per row (warp w: rows w, w + 16), then weights.  Lane j
  // keeps partial j's value (and j+32's) of the rows in registers.  These
  // loads go out ahead of the first partials', so the weights are worked
  // out while the partials arrive.
  constexpr int kRowsPerWarp = kCombineRows / kWarps;
  float x0[kRowsPerWarp], x1[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int lr = r0 + warp + kWarps * k;
    x0[k] = (lr < rows && lane < nseg) ? lse_part[(seg0 + lane) * rows + lr] : -INFINITY;
    x1[k] = (lr < rows && lane + 32 < nseg) ? lse_part[(seg0 + lane + 32) * rows + lr] : -INFINITY;
  }
  issue(0);
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int rr = warp + kWarps * k, lr = r0 + rr;
    float L = -INFINITY;
    if (lr < rows) {
      float mx = fmaxf(x0[k], x1[k]);
      for (int j = lane + 64; j < nseg; j += 32) mx = fmaxf(mx, lse_part[(seg0 + j) * rows + lr]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sum = 0.f;
      if (mx != -INFINITY) {
        sum = expf(x0[k] - mx) + expf(x1[k] - mx);
        for (int j = lane + 64; j < nseg; j += 32) sum += expf(lse_part[(seg0 + j) * rows + lr] - mx);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      L = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
      if (table) {
        if (lane < nseg) wts[lane][rr] = (L == -INFINITY) ? 0.f : expf(x0[k] - L);
        if (lane + 32 < nseg) wts[lane + 32][rr] = (L == -INFINITY) ? 0.f : expf(x1[k] - L);
      }
    }
    if (lane == 0) {
      lrow[rr] = L;
      if (lr < rows && lse_out && cz == 0) lse_out[(size_t)b * rows + lr] = L;
    }
  }
  __syncthreads();

  const float L = lrow[lane];
  float4 acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
  for (int j0 = 0; j0 < nseg; j0 += kBatch) {
    if (j0 > 0) issue(j0);
    if (valid && L != -INFINITY) {
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const int j = j0 + jj;
        const float w = j >= nseg ? 0.f : table ? wts[j][lane] : expf(lse_part[(seg0 + j) * rows + row] - L);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          acc[k].x += w * pv[jj][k].x; acc[k].y += w * pv[jj][k].y;
          acc[k].z += w * pv[jj][k].z; acc[k].w += w * pv[jj][k].w;
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    uint2 pk;
    pk.x = pack_bf16x2(acc[k].x, acc[k].y);
    pk.y = pack_bf16x2(acc[k].z, acc[k].w);
    *reinterpret_cast<uint2*>(&tile[lane][(warp + kWarps * k) * 4]) = pk;
  }
  __syncthreads();
  constexpr int kPieces = kCols * 2 / 16;  // 16-byte pieces per row
  for (int i = threadIdx.x; i < kCombineRows * kPieces; i += kThreads) {
    const int rr = i / kPieces, pc = i % kPieces;
    if (r0 + rr < rows)
      reinterpret_cast<uint4*>(o_lat + ((size_t)b * rows + r0 + rr) * DG + cz * kCols)[pc] =
          *reinterpret_cast<const uint4*>(&tile[rr][pc * 8]);
  }
}


// ---------------------------------------------------------------- combine + project
// One CTA of 512 threads per (head h, up to 64 query rows m = (b, l)).  The
// product is computed transposed, out^T = W_UV[h] . o_lat^T, so W_UV's 128
// output rows are the MMA's M and the CTA's query rows its N (rounded up to
// a multiple of 16): the CTA reads each weight once, and a small batch
// needs only a small merged tile.
//   * All of W_UV[h] is requested by TMA at once (DG/64 boxes of 128 rows x
//     64 columns, K-major, 128-byte swizzle), to land while the rows merge.
//   * The split plan of the CTA's sequences is read once into shared memory;
//     then the sixteen warps merge the rows (warp w: rows w, w + 16, ...;
//     lane i: the 8-column chunks i and i + 32), each row's partials and
//     log-sum-exps requested together, straight into the B tile (K-major,
//     128-byte swizzle: DG/64 boxes of N rows x 64 columns).
//   * One thread issues the DG/16 MMAs (M = 128, N, K = 16 each, fp32
//     accumulator in tensor memory); four warps (tensor-memory lane =
//     output dimension d) store out[m, h, d] as bf16, 64 contiguous bytes
//     per row m and warp.
// Optionally also writes o_lat (bf16) and the row log-sum-exp.
constexpr int kCpThreads = 512, kCpRows = 64;
template <int DG>
__global__ void __launch_bounds__(kCpThreads, 1)
    combine_project_kernel(const __grid_constant__ CUtensorMap tmA, const float* __restrict__ o_part,
                           const float* __restrict__ lse_part, const WsHeader* __restrict__ ws,
                           __nv_bfloat16* __restrict__ out, __nv_bfloat16* __restrict__ o_lat,
                           float* __restrict__ lse_out, int B, int Lq, int H, int G, int slots, int N) {
  constexpr int kBoxes = DG / 64;
  constexpr int kBoxA = kDhc * 64 * 2;  // 128 output rows x 64 latent columns, 16 KiB
  constexpr int kWarps = kCpThreads / 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sA = smem_u32(smem), sB = smem_u32(smem + kBoxes * kBoxA);
  const uint32_t boxB = (uint32_t)N * 128;  // one 64-column box of the B tile
  __shared__ __align__(8) uint64_t bars[2];  // W_UV landed, MMAs done
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int plan_s0[kCpRows], plan_n[kCpRows];  // slot range of the CTA's sequences
  const int h = blockIdx.x, m0 = blockIdx.y * kCpRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = Lq * H, M = B * Lq, g = (h * G) / H;
  const int mt = min(kCpRows, M - m0);  // query rows of this CTA (N = mt rounded up to 16)
  const int b0 = m0 / Lq, nb = (m0 + mt - 1) / Lq - b0 + 1;  // its sequences
  const uint32_t full = smem_u32(&bars[0]), done = smem_u32(&bars[1]);
  const uint32_t tcols = N <= 32 ? 32 : 64;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(full, 1);
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    // the weight tiles do not depend on the kernel before: start them now
    for (int q = 0; q < kBoxes; ++q) tma_prefetch_l2_3d(&tmA, 64 * q, 0, h);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(full, kBoxes * kBoxA);
    for (int q = 0; q < kBoxes; ++q) tma_load_3d(sA + q * kBoxA, &tmA, full, 64 * q, 0, h);
  }
  const bool plan_ok = ws->B == B;  // CTA-uniform
  if (plan_ok && threadIdx.x < nb) {
    const WsView v = ws_view(ws, B);
    const int s0 = v.slot0[b0 + threadIdx.x];
    plan_s0[threadIdx.x] = s0 < 0 ? 0 : s0;
    plan_n[threadIdx.x] = (s0 < 0 || s0 >= slots) ? 0 : min(v.nslot[b0 + threadIdx.x], slots - s0);
  }
  __syncthreads();

  // ---- merge the CTA's rows into the B tile
  if (plan_ok) {
    // 8-column chunks per lane and row: 2 or 1 (a 128- or 64-wide group latent
    // has fewer chunks than lanes; the spare lanes repeat chunks, which
    // writes the same values twice)
    constexpr int kLaneChunks = DG >= 256 ? DG / 8 / 32 : 1;
#pragma unroll 1
    for (int rr = warp; rr < mt; rr += kWarps) {
      const int m = m0 + rr, row = (m % Lq) * H + h;
      const int bi = m / Lq - b0;
      int chs[kLaneChunks];
#pragma unroll
      for (int i = 0; i < kLaneChunks; ++i) chs[i] = g * (DG / 8) + (lane + 32 * i) % (DG / 8);
      float4 acc[kLaneChunks][2];
      float L;
      merge_row(plan_s0[bi], plan_n[bi], o_part, lse_part, row, rows, chs, acc, L);
#pragma unroll
      for (int i = 0; i < kLaneChunks; ++i) {
        const int ch = (lane + 32 * i) % (DG / 8), box = ch >> 3, c8 = ch & 7;
        const uint32_t w0 = pack_bf16x2(acc[i][0].x, acc[i][0].y), w1 = pack_bf16x2(acc[i][0].z, acc[i][0].w);
        const uint32_t w2 = pack_bf16x2(acc[i][1].x, acc[i][1].y), w3 = pack_bf16x2(acc[i][1].z, acc[i][1].w);
        const uint32_t dst = sB + box * boxB + rr * 128 + ((c8 ^ (rr & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                     : "memory");
        if (o_lat) *reinterpret_cast<uint4*>(o_lat + ((size_t)m * H + h) * DG + 8 * ch) = make_uint4(w0, w1, w2, w3);
      }
      if (lane == 0 && lse_out) lse_out[(size_t)m * H + h] = L;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B tile: generic writes -> MMA reads
  __syncthreads();

  // ---- the product, one thread
  if (threadIdx.x == 0) {
    if (mbar_wait(full, 0, &abort_flag)) {  // W_UV always lands (it is waited for either way)
      if (plan_ok) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(kDhc, N, false, false);
#pragma unroll
        for (int kk = 0; kk < DG / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(sA + (kk >> 2) * kBoxA + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sB + (kk >> 2) * boxB + (kk & 3) * 32, 16, 1024);
          mma_ss(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
      }
      mma_commit(done);  // also arrives with no MMA issued
    } else {
      abort_flag = 1;
    }
  }
  __syncwarp();  // warp 0 reconverges before the aligned TMEM loads below
  if (warp < 4) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, &abort_flag));
    tc_fence_after();
    if (ok && plan_ok) {
      const int d = warp * 32 + lane;  // output dimension = tensor-memory lane
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int mm = c0 + k;
          if (mm < mt) out[((size_t)(m0 + mm) * H + h) * kDhc + d] = __float2bfloat16_rn(__uint_as_float(r[k]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// SMs of the current device (read once; every device this runs on is alike)
int device_sms() {
  static std::atomic<int> sms{0};
  int n = sms.load(std::memory_order_relaxed);
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 1;
    sms.store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int DG>
cudaError_t launch_combine_dg(const float* o_part, const float* lse_part, const WsHeader* ws, __nv_bfloat16* ol,
                              float* lse, int B, int Lq, int H, int G, int slots, cudaStream_t st) {
  constexpr int kCols = DG < kCombineCols ? DG : kCombineCols;
  dim3 grid(B, (Lq * H + kCombineRows - 1) / kCombineRows, DG / kCols);
  if ((long long)grid.x * grid.y * grid.z > device_sms())  // more than one wave: two CTAs an SM
    combine_kernel<DG, kCombineThreads / 2, 2><<<grid, kCombineThreads / 2, 0, st>>>(o_part, lse_part, ws, ol, lse,
                                                                                    B, Lq, H, G, slots);
  else
    combine_kernel<DG, kCombineThreads, 4><<<grid, kCombineThreads, 0, st>>>(o_part, lse_part, ws, ol, lse, B, Lq,
                                                                            H, G, slots);
  return cudaGetLastError();
}
template <int DG>
cudaError_t launch_combine_project_dg(const CUtensorMap& tmA, const float* o_part, const float* lse_part,
                                      const WsHeader* ws, __nv_bfloat16* o, __nv_bfloat16* ol, float* lse, int B,
                                      int Lq, int H, int G, int slots, cudaStream_t st) {
  const int M = B * Lq;
  const int mt = M < kCpRows ? M : kCpRows;
  const int N = (mt + 15) / 16 * 16;
  dim3 grid(H, (M + kCpRows - 1) / kCpRows);
  const int smem = (DG / 64) * kDhc * 64 * 2 + N * DG * 2 + 1024;
  const int smem_max = (DG / 64) * kDhc * 64 * 2 + kCpRows * DG * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(combine_project_kernel<DG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  if (e != cudaSuccess) return e;
  // launched plainly (like the combine): chained, its CTAs wait on the SMs
  // of work units that finished early, and the step measured slower
  combine_project_kernel<DG><<<grid, kCpThreads, smem, st>>>(tmA, o_part, lse_part, ws, o, ol, lse, B, Lq, H, G,
                                                             slots, N);
  return cudaGetLastError();
}

}  // namespace

// The combine is launched plainly, not chained to the decode: chained, its
// CTAs become resident early on the SMs of work units that had no pages and
// wait there, and the step measured 1-2 us slower on every workload.  (Its
// griddepcontrol calls are then no-ops; the projection after it is still
// chained.)
cudaError_t launch_combine(const float* o_part, const float* lse_part, const WsHeader* ws, void* o_lat,
                           float* lse, int B, int Lq, int H, int G, int slots, cudaStream_t st) {
  auto* ol = static_cast<__nv_bfloat16*>(o_lat);
  switch (kDc / G) {
    case 512: return launch_combine_dg<512>(o_part, lse_part, ws, ol, lse, B, Lq, H, G, slots, st);
    case 256: return launch_combine_dg<256>(o_part, lse_part, ws, ol, lse, B, Lq, H, G, slots, st);
    case 128: return launch_combine_dg<128>(o_part, lse_part, ws, ol, lse, B, Lq, H, G, slots, st);
    case 64: return launch_combine_dg<64>(o_part, lse_part, ws, ol, lse, B, Lq, H, G, slots, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_project(const CUtensorMap& tmA, const float* o_part, const float* lse_part,
                                   const WsHeader* ws, void* out, void* o_lat, float* lse, int B, int Lq, int H,
                                   int G, int slots, cudaStream_t st) {
  auto* o = static_cast<__nv_bfloat16*>(out);
  auto* ol = static_cast<__nv_bfloat16*>(o_lat);
  switch (kDc / G) {
    case 512: return launch_combine_project_dg<512>(tmA, o_part, lse_part, ws, o, ol, lse, B, Lq, H, G, slots, st);
    case 256: return launch_combine_project_dg<256>(tmA, o_part, lse_part, ws, o, ol, lse, B, Lq, H, G, slots, st);
    case 128: return launch_combine_project_dg<128>(tmA, o_part, lse_part, ws, o, ol, lse, B, Lq, H, G, slots, st);
    case 64: return launch_combine_project_dg<64>(tmA, o_part, lse_part, ws, o, ol, lse, B, Lq, H, G, slots, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
