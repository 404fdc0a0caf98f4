// mla_gemm.cu — the two per-head batched GEMMs around the attention kernel,
// on the tcgen05 tensor cores (operands staged by TMA, fp32 accumulator in
// tensor memory).
//
//   absorb : q_cat[m,h,0:d_g] = q_nope[m,h,:] . W_UK[h]      (M x 128 x d_g per head)
//            q_cat[m,h,d_g:]  = q_rope[m,h,:]
//            (matrix absorption, MLA operator write-up §4, einsum qhd,hdc->qhc)
//   project: out[m,h,:]       = W_UV[h] . o_lat[m,h,:]        (M x d_g x 128 per head)
//
// m runs over the B*Lq query rows.  absorb: one CTA per (head, 128-row
// block, up to 256 output columns); project: one CTA per (head, 128-row
// block, 64 output columns).
// Rows past M are zero-filled by the tensor copies and never stored.
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Store 32 fp32 accumulator columns of one row as bf16 (64 bytes).
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
    v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
    v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
    v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
    d[q] = v;
  }
}

constexpr int kBox = 16384;  // one 128 x 64 bf16 tile, 128-byte swizzled

// ---------------------------------------------------------------- absorb
// A = q_nope rows (K-major, 2 tiles of 64 k), B = kCols = min(256, d_g)
// columns of W_UK[h] (d rows x c columns, N-contiguous, i.e. MN-major:
// kCols/64 tiles of 128 d x 64 c).  Two CTAs per SM, all resident at once:
// the weight loads of one overlap the MMAs and stores of the other.
constexpr int kAbsorbCols = 256;
__host__ __device__ constexpr int absorb_cols(int dg) { return dg < kAbsorbCols ? dg : kAbsorbCols; }
template <int DG>
__global__ void __launch_bounds__(128)
    absorb_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __nv_bfloat16* __restrict__ q_rope, __nv_bfloat16* __restrict__ q_cat,
                  int M, int H) {
  constexpr int kCols = absorb_cols(DG);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + 2 * kBox;
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  const int h = blockIdx.x, m0 = blockIdx.y * kRowsPerCta, n0 = blockIdx.z * kCols;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full = smem_u32(&bars[0]), done = smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(full, 1);
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // the weight tiles do not depend on the kernel before: start them now
    for (int nb = 0; nb < kCols / 64; ++nb) tma_prefetch_l2_3d(&tmB, n0 + nb * 64, 0, h);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  // set-up above overlaps the kernel before; global memory only from here on
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(full, 2 * kBox + (kCols / 64) * kBox);
    for (int nb = 0; nb < kCols / 64; ++nb)
      tma_load_3d(smem_u32(sB + nb * kBox), &tmB, full, n0 + nb * 64, 0, h);
    for (int kb = 0; kb < 2; ++kb) tma_load_3d(smem_u32(sA + kb * kBox), &tmA, full, kb * 64, h, m0);
    if (mbar_wait(full, 0, &abort_flag)) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(128, kCols, false, true);
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // K = 128 in steps of 16
        const uint64_t ad = sdesc_sw128(smem_u32(sA) + (j >> 2) * kBox + (j & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(smem_u32(sB) + j * 2048, kBox, 1024);  // 64-column atoms kBox apart
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
  if (ok) {
    const int row = warp * 32 + lane, m = m0 + row;
    __nv_bfloat16* dst = q_cat + ((size_t)m * H + h) * (DG + kDr);
#pragma unroll 1
    for (int c = 0; c < kCols / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
      tmem_wait_ld();
      if (m < M) store_row32_bf16(dst + n0 + c * 32, r);
    }
    if (m < M && blockIdx.z == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(q_rope + ((size_t)m * H + h) * kDr);
      uint4* d = reinterpret_cast<uint4*>(dst + DG);
#pragma unroll
      for (int q = 0; q < kDr * 2 / 16; ++q) d[q] = src[q];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ---------------------------------------------------------------- project
// A = o_lat rows (K-major over d_g), B = 64 rows of W_UV[h] (d rows x d_g
// columns, K-contiguous: K-major).  K is streamed in 64-wide chunks through
// a 4-slot ring; each slot holds one A tile (16 KiB) and one B tile (8 KiB).
// Two CTAs per head (output columns 0-63, 64-127), two CTAs per SM.
constexpr int kProjectCols = 64;
template <int DG>
__global__ void __launch_bounds__(128)
    project_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   __nv_bfloat16* __restrict__ out, int M, int H) {
  constexpr int kSlots = 4, kChunks = DG / 64, kBoxB = kProjectCols * 64 * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(8) uint64_t bars[2 * kSlots + 1];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  const int h = blockIdx.x, m0 = blockIdx.y * kRowsPerCta, n0 = blockIdx.z * kProjectCols;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t done = smem_u32(&bars[2 * kSlots]);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kSlots + s]); };
  auto slotA = [&](int s) { return smem_u32(smem + s * (kBox + kBoxB)); };
  auto slotB = [&](int s) { return smem_u32(smem + s * (kBox + kBoxB) + kBox); };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // the weight tiles do not depend on the kernel before: start them now
    for (int c = 0; c < kChunks; ++c) tma_prefetch_l2_3d(&tmB, c * 64, n0, h);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_holder), kProjectCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  // set-up above overlaps the kernel before; global memory only from here on
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    auto load = [&](int c) {
      const int s = c % kSlots;
      mbar_arrive_expect_tx(full(s), kBox + kBoxB);
      tma_load_3d(slotB(s), &tmB, full(s), c * 64, n0, h);
      tma_load_3d(slotA(s), &tmA, full(s), c * 64, h, m0);
    };
    for (int c = 0; c < kChunks && c < kSlots; ++c) load(c);
    constexpr uint32_t idesc = idesc_bf16(128, kProjectCols, false, false);
    bool ok = true;
    for (int c = 0; c < kChunks && ok; ++c) {
      const int s = c % kSlots;
      if (!(ok = mbar_wait(full(s), (c / kSlots) & 1, &abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t ad = sdesc_sw128(slotA(s) + j * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(slotB(s) + j * 32, 16, 1024);
        mma_ss(tmem, ad, bd, idesc, (c > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit(empty(s));
      if (c + kSlots < kChunks) {
        if (!(ok = mbar_wait(empty(s), (c / kSlots) & 1, &abort_flag))) break;
        load(c + kSlots);
      }
    }
    if (ok) mma_commit(done);
    else abort_flag = 1;
  }
  __syncwarp();  // warp 0 reconverges before the aligned TMEM loads below
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, &abort_flag));
  tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane, m = m0 + row;
    __nv_bfloat16* dst = out + ((size_t)m * H + h) * kDhc + n0;
#pragma unroll 1
    for (int c = 0; c < kProjectCols / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
      tmem_wait_ld();
      if (m < M) store_row32_bf16(dst + c * 32, r);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kProjectCols);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

template <int DG>
cudaError_t launch_absorb_dg(const CUtensorMap& tmA, const CUtensorMap& tmB, const __nv_bfloat16* qr,
                             __nv_bfloat16* qc, int M, int H, cudaStream_t st) {
  constexpr int kCols = absorb_cols(DG);
  dim3 grid(H, (M + kRowsPerCta - 1) / kRowsPerCta, DG / kCols), block(128);
  const int smem = 2 * kBox + (kCols / 64) * kBox + 1024;
  cudaError_t e = set_smem(absorb_kernel<DG>, smem);
  if (e != cudaSuccess) return e;
  return launch_chained(absorb_kernel<DG>, grid, block, smem, st, tmA, tmB, qr, qc, M, H);
}
template <int DG>
cudaError_t launch_project_dg(const CUtensorMap& tmA, const CUtensorMap& tmB, __nv_bfloat16* o, int M, int H,
                              cudaStream_t st) {
  dim3 grid(H, (M + kRowsPerCta - 1) / kRowsPerCta, kDhc / kProjectCols), block(128);
  const int smem = 4 * (kBox + kProjectCols * 64 * 2) + 1024;
  cudaError_t e = set_smem(project_kernel<DG>, smem);
  if (e != cudaSuccess) return e;
  return launch_chained(project_kernel<DG>, grid, block, smem, st, tmA, tmB, o, M, H);
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
