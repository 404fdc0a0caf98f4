// mla_combine.cu — log-sum-exp merge of the split-KV partials written by the
// decode kernel into the latent output o_lat (bf16) and the row log-sum-exp.
//
// The MLA pages name split-KV decoding but give no merge; this is the exact
// identity of a softmax taken over disjoint key ranges.  A split s of a query
// row holds o_s = (sum_k p_k v_k) / l_s and lse_s = m_s + log l_s over its
// keys; the row's result is L = log sum_s exp(lse_s) and
// o = sum_s exp(lse_s - L) o_s.  Splits with no keys carry lse = -inf and
// weigh nothing.  The partials are chunk-major, [slot][column/4][row][4];
// sequence b owns slots slot0[b] .. slot0[b] + nslot[b] - 1 of the workspace.
#include <cmath>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

// ---------------------------------------------------------------- combine
// One CTA of 512 threads per (sequence, 32 query rows, 256 latent columns):
// one CTA fits an SM at a time, so a grid of about one CTA per SM finishes
// in one wave.  The first partials' loads are issued before the row
// weights are known, so the CTA waits for two dependent global round trips
// (split records, then log-sum-exps and partials together), not three.
// The log-sum-exp of each row's partials is reduced with warp shuffles over
// the partial index and turned into per-partial weights in shared memory;
// the weighted sum reads the chunk-major partials coalesced (32 consecutive
// rows per warp access).  The bf16 result is staged in shared memory and
// written out as contiguous row pieces.
constexpr int kCombineRows = 32, kCombineCols = 256, kCombineMaxSeg = 64, kCombineThreads = 512;
template <int DG>
__global__ void __launch_bounds__(kCombineThreads, 1)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                   const WsHeader* __restrict__ ws, __nv_bfloat16* __restrict__ o_lat,
                   float* __restrict__ lse_out, int B, int Lq, int H, int G) {
  constexpr int kCols = kCombineCols;  // columns of this CTA
  constexpr int kWarps = kCombineThreads / 32;
  static_assert(DG % kCols == 0, "latent slice in whole CTA column ranges");
  __shared__ __align__(16) __nv_bfloat16 tile[kCombineRows][kCols + 8];
  __shared__ float wts[kCombineMaxSeg][kCombineRows];
  __shared__ float lrow[kCombineRows];
  const int rows = Lq * H;
  const int b = blockIdx.x, r0 = blockIdx.y * kCombineRows, cz = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  const WsView v = ws_view(ws, B);
  const int nseg = v.nslot[b];
  const size_t seg0 = (size_t)v.slot0[b];
  const bool table = nseg <= kCombineMaxSeg;

  // weighted-sum thread layout: (row lane, chunk group warp); the first
  // kBatch partials of the thread's chunks are requested right away
  const int row = r0 + lane;
  const bool valid = row < rows;
  const int h = valid ? row % H : 0, g = (h * G) / H;
  constexpr int kChunks = kCols / 4, kPer = kChunks / kWarps;  // chunks of this thread: warp + kWarps*k
  constexpr int kBatch = 4;  // partials whose loads are all issued before any is used
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
  issue(0);

  // log-sum-exp per row (warp w: rows w, w + 16), then weights.  Lane j
  // keeps partial j's value (and j+32's) of the rows in registers.
  constexpr int kRowsPerWarp = kCombineRows / kWarps;
  float x0[kRowsPerWarp], x1[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int lr = r0 + warp + kWarps * k;
    x0[k] = (lr < rows && lane < nseg) ? lse_part[(seg0 + lane) * rows + lr] : -INFINITY;
    x1[k] = (lr < rows && lane + 32 < nseg) ? lse_part[(seg0 + lane + 32) * rows + lr] : -INFINITY;
  }
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
  for (int i = threadIdx.x; i < kCombineRows * kPieces; i += kCombineThreads) {
    const int rr = i / kPieces, pc = i % kPieces;
    if (r0 + rr < rows)
      reinterpret_cast<uint4*>(o_lat + ((size_t)b * rows + r0 + rr) * DG + cz * kCols)[pc] =
          *reinterpret_cast<const uint4*>(&tile[rr][pc * 8]);
  }
}

}  // namespace

// The combine is launched plainly, not chained to the decode: chained, its
// CTAs become resident early on the SMs of work units that had no pages and
// wait there, and the step measured 1-2 us slower on every workload.  (Its
// griddepcontrol calls are then no-ops; the projection after it is still
// chained.)
cudaError_t launch_combine(const float* o_part, const float* lse_part, const WsHeader* ws, void* o_lat,
                           float* lse, int B, int Lq, int H, int G, cudaStream_t st) {
  const int d_g = kDc / G;
  dim3 grid(B, (Lq * H + kCombineRows - 1) / kCombineRows, d_g / kCombineCols), block(kCombineThreads);
  auto* ol = static_cast<__nv_bfloat16*>(o_lat);
  if (G == 1) combine_kernel<512><<<grid, block, 0, st>>>(o_part, lse_part, ws, ol, lse, B, Lq, H, G);
  else combine_kernel<256><<<grid, block, 0, st>>>(o_part, lse_part, ws, ol, lse, B, Lq, H, G);
  return cudaGetLastError();
}

}  // namespace mla
