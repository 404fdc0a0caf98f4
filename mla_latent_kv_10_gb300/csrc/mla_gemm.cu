// mla_gemm.cu — the two per-head batched GEMMs around the attention kernel,
// on the tcgen05 tensor cores (operands staged by TMA, fp32 accumulator in
// tensor memory).
//
//   absorb : q_cat[m,h,0:d_g] = q_nope[m,h,:] . W_UK[h]      (M x 128 x d_g per head)
//            q_cat[m,h,d_g:]  = q_rope[m,h,:]
//            (matrix absorption, MLA operator write-up §4, einsum qhd,hdc->qhc)
//   project: out[m,h,:]       = W_UV[h] . o_lat[m,h,:]        (M x d_g x 128 per head)
//
// Both products run transposed, with the weight as the MMA's A operand and
// the query rows as its N: M = 128 weight columns (absorb: output latents c;
// project: output dimensions d), N = the B*Lq query rows of the CTA rounded
// up to 16 (at most 128).  A decode batch has few query rows (16 on the
// DeepSeek-V3 decode), and as the A operand they would fill a 128-row tile
// mostly with zeros; as N they cost what they hold.  The accumulator then
// holds D^T (tensor-memory lane = output column, column = query row); the
// epilogue turns it back through shared memory and writes whole row pieces.
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int kBox = 16384;              // one 64-column x 128-row bf16 tile, 128-byte swizzled
constexpr int kTilePitch = kDhc + 8;     // bf16 elements per row of the epilogue's transposed tile
__host__ __device__ constexpr int rows_n(int M) {  // the MMA's N: query rows per CTA, rounded up to 16
  return ((M < kRowsPerCta ? M : kRowsPerCta) + 15) / 16 * 16;
}
__host__ __device__ constexpr uint32_t tmem_cols_for(int n) { return n <= 32 ? 32 : n <= 64 ? 64 : 128; }

// The transposed epilogue.  Tensor memory holds D^T for 128 output columns
// (lane) and N query rows (column).  Each warp reads its 32 lanes 16 columns
// at a time and writes them into the bf16 tile [row][column] in shared
// memory (a warp's 32 lanes fill 64 contiguous bytes of one row); then the
// block writes each valid row's first `ncols` columns to dst_row(m) as
// 16-byte pieces.
template <typename RowPtr>
__device__ __forceinline__ void store_transposed(uint32_t tmem, int N, int rows_valid, int ncols,
                                                 __nv_bfloat16* tile, RowPtr dst_row) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, col = warp * 32 + lane;
#pragma unroll 1
  for (int c0 = 0; c0 < N; c0 += 16) {
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 16; ++k) tile[(c0 + k) * kTilePitch + col] = __float2bfloat16_rn(__uint_as_float(r[k]));
  }
  __syncthreads();
  const int pieces = ncols / 8;
  for (int i = threadIdx.x; i < rows_valid * pieces; i += blockDim.x) {
    const int m = i / pieces, pc = i % pieces;
    reinterpret_cast<uint4*>(dst_row(m))[pc] = *reinterpret_cast<const uint4*>(tile + m * kTilePitch + pc * 8);
  }
}

// ---------------------------------------------------------------- absorb
// One CTA per (head h, block of up to 128 query rows, 128 output latents
// n0..n0+127).  A = W_UK[h][:, n0:n0+128] (d rows x c columns, c
// contiguous: MN-major, two 64-column tiles of 128 d); B = the rows'
// q_nope[m, h, :] (K-major, two 64-wide tiles of N rows).  K = d_hc = 128.
// Small: up to four CTAs per SM.
template <int DG>
__global__ void __launch_bounds__(128)
    absorb_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __nv_bfloat16* __restrict__ q_rope, __nv_bfloat16* __restrict__ q_cat,
                  int M, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int N = rows_n(M), boxQ = N * 128;
  const uint32_t sW = smem_u32(smem), sQ = sW + 2 * kBox;
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  const int h = blockIdx.x, m0 = blockIdx.y * kRowsPerCta, n0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5;
  const uint32_t full = smem_u32(&bars[0]), done = smem_u32(&bars[1]);
  const uint32_t tcols = tmem_cols_for(N);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(full, 1);
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // The weight is no kernel's output, so its tiles are requested before
    // the wait for the kernel before (whose tail they overlap).  DG = 64:
    // one W tile; A's rows 64..127 are then left as they are, and the
    // accumulator lanes they produce are never stored.
    const int nW = DG - n0 >= 128 ? 2 : 1;
    mbar_arrive_expect_tx(full, nW * kBox + 2 * boxQ);
    for (int t = 0; t < nW; ++t) tma_load_3d(sW + t * kBox, &tmB, full, n0 + 64 * t, 0, h);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  // global memory the kernels before may write only from here on
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int kb = 0; kb < 2; ++kb) tma_load_3d(sQ + kb * boxQ, &tmA, full, kb * 64, h, m0);
    if (mbar_wait(full, 0, &abort_flag)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, N, true, false);
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // K = 128 in steps of 16
        const uint64_t ad = sdesc_sw128(sW + j * 2048, kBox, 1024);  // 64-column atoms kBox apart
        const uint64_t bd = sdesc_sw128(sQ + (j >> 2) * boxQ + (j & 3) * 32, 16, 1024);
        mma_ss(tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
      }
      mma_commit(done);
    } else {
      abort_flag = 1;
    }
  }
  __syncwarp();  // warp 0 reconverges before the aligned TMEM loads below
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, &abort_flag));
  tc_fence_after();
  const int rows_valid = min(N, M - m0);
  // the operand tiles are dead once the MMAs completed: the transposed tile reuses them
  if (__syncthreads_and(ok)) {
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem);
    store_transposed(tmem, N, rows_valid, min(128, DG - n0), tile,
                     [&](int m) { return q_cat + ((size_t)(m0 + m) * H + h) * (DG + kDr) + n0; });
    if (blockIdx.z == 0) {  // q_cat[m, h, DG:] = q_rope[m, h, :]
      constexpr int kP = kDr * 2 / 16;
      for (int i = threadIdx.x; i < rows_valid * kP; i += blockDim.x) {
        const int m = m0 + i / kP, q = i % kP;
        reinterpret_cast<uint4*>(q_cat + ((size_t)m * H + h) * (DG + kDr) + DG)[q] =
            reinterpret_cast<const uint4*>(q_rope + ((size_t)m * H + h) * kDr)[q];
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

// ---------------------------------------------------------------- project
// One CTA per (head h, block of up to 128 query rows), all 128 output
// dimensions.  A = W_UV[h] (d rows x c columns, c contiguous: K-major), B =
// the rows' o_lat[m, h, :] (K-major).  K = DG streamed in 64-wide chunks
// through `slots` ring slots (each one 128 x 64 tile of W_UV and one N x 64
// tile of o_lat); when every chunk fits, all are requested at once.
template <int DG>
__global__ void __launch_bounds__(128)
    project_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   __nv_bfloat16* __restrict__ out, int M, int H, int slots) {
  constexpr int kChunks = DG / 64, kMaxSlots = 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int N = rows_n(M), boxO = N * 128, slot_bytes = kBox + boxO;
  __shared__ __align__(8) uint64_t bars[2 * kMaxSlots + 1];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  const int h = blockIdx.x, m0 = blockIdx.y * kRowsPerCta;
  const int warp = threadIdx.x >> 5;
  const uint32_t done = smem_u32(&bars[2 * kMaxSlots]);
  const uint32_t tcols = tmem_cols_for(N);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kMaxSlots + s]); };
  auto slotW = [&](int s) { return smem_u32(smem + s * slot_bytes); };
  auto slotO = [&](int s) { return smem_u32(smem + s * slot_bytes + kBox); };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < slots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // The weight is no kernel's output: the W tiles of the ring's first
    // pass are requested before the wait for the kernel before (each
    // slot's barrier counts its W and o_lat tiles), the later ones go to
    // L2 now.
    for (int c = 0; c < kChunks; ++c) {
      if (c < slots) {
        mbar_arrive_expect_tx(full(c), slot_bytes);
        tma_load_3d(slotW(c), &tmB, full(c), c * 64, 0, h);
      } else {
        tma_prefetch_l2_3d(&tmB, c * 64, 0, h);
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  // global memory the kernels before may write only from here on
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    auto load = [&](int c) {
      const int s = c % slots;
      mbar_arrive_expect_tx(full(s), slot_bytes);
      tma_load_3d(slotW(s), &tmB, full(s), c * 64, 0, h);
      tma_load_3d(slotO(s), &tmA, full(s), c * 64, h, m0);
    };
    for (int c = 0; c < kChunks && c < slots; ++c) tma_load_3d(slotO(c), &tmA, full(c), c * 64, h, m0);
    const uint32_t idesc = idesc_bf16(128, N, false, false);
    bool ok = true;
    for (int c = 0; c < kChunks && ok; ++c) {
      const int s = c % slots, ph = (c / slots) & 1;
      if (!(ok = mbar_wait(full(s), ph, &abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t ad = sdesc_sw128(slotW(s) + j * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(slotO(s) + j * 32, 16, 1024);
        mma_ss(tmem, ad, bd, idesc, (c > 0 || j > 0) ? 1u : 0u);
      }
      if (c + slots < kChunks) {
        mma_commit(empty(s));
        if (!(ok = mbar_wait(empty(s), ph, &abort_flag))) break;
        load(c + slots);
      }
    }
    if (ok) mma_commit(done);
    else abort_flag = 1;
  }
  __syncwarp();  // warp 0 reconverges before the aligned TMEM loads below
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, &abort_flag));
  tc_fence_after();
  // the ring is dead once the MMAs completed: the transposed tile reuses it
  if (__syncthreads_and(ok)) {
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem);
    store_transposed(tmem, N, min(N, M - m0), kDhc, tile,
                     [&](int m) { return out + ((size_t)(m0 + m) * H + h) * kDhc; });
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

constexpr int kProjectSmemBudget = 200 * 1024;

}  // namespace

// The tensor maps: absorb tmA = q_nope (d, h, m) with 64 x 1 x rows_n(M)
// boxes, tmB = W_UK (c, d, h) with 64 x 128 x 1 boxes; project tmA = o_lat
// (c, h, m) with 64 x 1 x rows_n(M) boxes, tmB = W_UV (c, d, h) with
// 64 x 128 x 1 boxes.
int gemm_rows_box(int M) { return rows_n(M); }

template <int DG>
cudaError_t launch_absorb_dg(const CUtensorMap& tmA, const CUtensorMap& tmB, const __nv_bfloat16* qr,
                             __nv_bfloat16* qc, int M, int H, cudaStream_t st) {
  dim3 grid(H, (M + kRowsPerCta - 1) / kRowsPerCta, (DG + 127) / 128), block(128);
  const int N = rows_n(M);
  const int smem = 2 * kBox + 2 * N * 128 + 1024;  // >= the transposed tile, N x kTilePitch x 2 bytes
  cudaError_t e = set_smem(absorb_kernel<DG>, smem);
  if (e != cudaSuccess) return e;
  return launch_chained(absorb_kernel<DG>, grid, block, smem, st, tmA, tmB, qr, qc, M, H);
}
template <int DG>
cudaError_t launch_project_dg(const CUtensorMap& tmA, const CUtensorMap& tmB, __nv_bfloat16* o, int M, int H,
                              cudaStream_t st) {
  dim3 grid(H, (M + kRowsPerCta - 1) / kRowsPerCta), block(128);
  const int N = rows_n(M), slot_bytes = kBox + N * 128;
  int slots = kProjectSmemBudget / slot_bytes;
  if (slots > DG / 64) slots = DG / 64;
  const int ring = slots * slot_bytes, tile = N * kTilePitch * 2;
  const int smem = (ring > tile ? ring : tile) + 1024;
  cudaError_t e = set_smem(project_kernel<DG>, smem);
  if (e != cudaSuccess) return e;
  return launch_chained(project_kernel<DG>, grid, block, smem, st, tmA, tmB, o, M, H, slots);
}

cudaError_t launch_absorb(const CUtensorMap& tmA, const CUtensorMap& tmB, const void* q_rope,
                          void* q_cat, int M, int H, int d_g, cudaStream_t st) {
  const auto* qr = static_cast<const __nv_bfloat16*>(q_rope);
  auto* qc = static_cast<__nv_bfloat16*>(q_cat);
  switch (d_g) {
    case 512: return launch_absorb_dg<512>(tmA, tmB, qr, qc, M, H, st);
    case 256: return launch_absorb_dg<256>(tmA, tmB, qr, qc, M, H, st);
    case 128: return launch_absorb_dg<128>(tmA, tmB, qr, qc, M, H, st);
    case 64: return launch_absorb_dg<64>(tmA, tmB, qr, qc, M, H, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_project(const CUtensorMap& tmA, const CUtensorMap& tmB, void* out, int M, int H,
                           int d_g, cudaStream_t st) {
  auto* o = static_cast<__nv_bfloat16*>(out);
  switch (d_g) {
    case 512: return launch_project_dg<512>(tmA, tmB, o, M, H, st);
    case 256: return launch_project_dg<256>(tmA, tmB, o, M, H, st);
    case 128: return launch_project_dg<128>(tmA, tmB, o, M, H, st);
    case 64: return launch_project_dg<64>(tmA, tmB, o, M, H, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
