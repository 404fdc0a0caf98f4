// mla_internal.h — declarations shared by the kernels and the C-ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla.h"

namespace mla {

constexpr int kPage = 64;      // tokens per cache page
constexpr int kDc = 512;       // latent width (all groups)
constexpr int kDr = 64;        // RoPE key width
constexpr int kRow = kDc + kDr;  // 576 elements per cache row
constexpr int kDhc = 128;      // content head dim
constexpr int kRowsPerCta = 128;  // query rows (l, h) per CTA = MMA M
// FP8 cache row (bytes): 512 e4m3 codes | 64 bf16 RoPE key | 4 fp32 scales
constexpr int kFp8RopeByte = 512, kFp8ScaleByte = 640, kRowBytesFp8 = 656;

// Decode workspace: a 32-byte header, then int arrays
//   off[B+1]   page offset of each sequence in the flattened page order
//              (off[B] = total pages)
//   nlen[B]    validated sequence lengths
//   slot0[B]   first partial-output slot of sequence b
//   nslot[B]   number of partial-output slots of sequence b
//   rec[kMaxUnits]  one UnitRec per work unit (written by the plan kernel
//              when the decode kernel does not plan for itself)
// Split modes: 0 = balanced (the flattened page list cut into equal
// contiguous ranges, a range may cover several sequences; slot = b + unit),
// 1 = sequence-aligned (every unit inside one sequence; slot = unit).
constexpr int kMaxUnits = 256;
struct WsHeader {
  int status;    // sticky device status (mla_status), 0 = ok
  int total;     // total pages over all sequences
  int chunk;     // pages per work unit (balanced split)
  int units;     // work units (CTA clusters) of the last launch
  int B;
  int mode;      // 0 balanced, 1 sequence-aligned
  int pad[2];
};
static_assert(sizeof(WsHeader) == 32, "header layout");

// The pages one work unit decodes: starting at sequence b, whose first page
// sits at flattened offset o, the unit covers flattened pages [start, end)
// (sequence-aligned split: o = 0 and [start, end) are pages of sequence b).
// The partial of a segment of sequence sb goes to slot sb + bias.
struct UnitRec {
  int b, o, start, end, bias;
};

struct WsView {
  int *off, *nlen, *slot0, *nslot;
  UnitRec* rec;
};
__host__ __device__ inline WsView ws_view(const WsHeader* ws, int B) {
  int* p = const_cast<int*>(reinterpret_cast<const int*>(ws + 1));
  WsView v;
  v.off = p;
  v.nlen = v.off + B + 1;
  v.slot0 = v.nlen + B;
  v.nslot = v.slot0 + B;
  v.rec = reinterpret_cast<UnitRec*>(v.nslot + B);
  return v;
}

inline size_t ws_bytes_for(int B) {
  size_t b = sizeof(WsHeader) + sizeof(int) * ((size_t)4 * B + 1) + sizeof(UnitRec) * kMaxUnits;
  return (b + 255) & ~(size_t)255;
}

struct DecodeArgs {
  const __nv_bfloat16* q_cat;
  const int32_t* block_table;
  float* o_part;
  float* lse_part;
  WsHeader* ws;
  int B, Lq, H, G, d_g, max_pages, num_pages, causal, rows;  // rows = Lq*H
  float scale_log2;   // scale * log2(e)
  int plan_in_kernel; // 1: every CTA computes the split itself (B <= decode_plan_max_b)
  int units;
  const int32_t* seq_lens;
  unsigned long long wait_ns;  // wall-clock limit of each pipeline wait inside the kernel
  int stall_page;              // testing: the QK issuer waits on a barrier nothing completes before this page (-1: off)
};
// Testing settings of the decode launches (mla_set_timeout_test): the limit
// of the pipeline waits (normally 2 s) and the page before which the QK
// issuer stalls (normally -1, never).
unsigned long long decode_wait_limit_ns();
int decode_stall_page();
// the decode kernel plans its own split for batches up to these sizes (one
// sequence a thread; its blocks have 512 threads in pair mode, for one
// latent group, and 352 in solo mode, for grouped latents, 384 with an FP8
// cache)
constexpr int kPlanInKernelMaxB = 448, kPlanInKernelMaxBSolo = 352;

// launchers (return cudaError_t of the launch)
cudaError_t launch_absorb(const CUtensorMap& tmA, const CUtensorMap& tmB, const void* q_rope,
                          void* q_cat, int M, int H, int d_g, cudaStream_t st);
cudaError_t launch_project(const CUtensorMap& tmA, const CUtensorMap& tmB, void* out, int M, int H,
                           int d_g, cudaStream_t st);
cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* block_table, WsHeader* ws, int B,
                        int Lq, int max_pages, int num_pages, int units, cudaStream_t st);
// tm_cache: latent boxes (64 x 64, 128-byte swizzle); tm_rope: the cache's
// RoPE columns (32 x 64 boxes, 64-byte swizzle); tm_qrope: q_cat rows
// (32 x 128 boxes, 64-byte swizzle); tm_qlat: q_cat rows (64 x 128 boxes,
// 128-byte swizzle)
// solo: the kernel mode for 2, 4 or 8 latent groups (each CTA of a pair
// serves the heads of its latent half, no exchange; tm_qrope then has boxes
// of 32 x H/2); otherwise the pair mode for one group.
// fp8: the cache rows are FP8 (kRowBytesFp8 bytes): tm_cache then holds
// the codes as bytes (64 x 64 boxes, no swizzle), tm_rope the RoPE key as
// bf16 of the same rows, tm_scale the scales as fp32 (4 x 64 boxes); in
// bf16 mode tm_scale is not read.
cudaError_t launch_decode(bool solo, bool fp8, const CUtensorMap& tm_cache, const CUtensorMap& tm_rope,
                          const CUtensorMap& tm_qrope, const CUtensorMap& tm_qlat, const CUtensorMap& tm_scale,
                          const DecodeArgs& a, int units, int csize, cudaStream_t st);
// Launch with programmatic stream serialization: the kernel may start its
// set-up while the kernel before it on the stream finishes (every kernel of
// this library waits for its predecessor before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// slots: partial slots the caller allocated (bounds every slot range read)
cudaError_t launch_combine(const float* o_part, const float* lse_part, const WsHeader* ws,
                           void* o_lat, float* lse, int B, int Lq, int H, int G, int slots, cudaStream_t st);
// tmA: W_UV in 64-column boxes of one head's 128 rows
cudaError_t launch_combine_project(const CUtensorMap& tmA, const float* o_part, const float* lse_part,
                                   const WsHeader* ws, void* out, void* o_lat, float* lse, int B, int Lq, int H,
                                   int G, int slots, cudaStream_t st);
int decode_max_units(bool solo, bool fp8, int csize, int* units);  // clusters of csize CTAs resident at once
// The decompress branch (mla_prefill.cu).  tmC: cache rows (64 x 64 boxes,
// 128-byte swizzle); tmWK, tmWV: W_UK, W_UV as [H, 128, d_g] (64 x 128 x 1
// boxes); tmQN, tmQR: q_nope, q_rope as [B*Lq rows, H*128 / H*64 columns]
// (64 x 128 boxes); tmK, tmV: k_nope, v as [B*H*S rows, 128 columns]
// (64 x 64 boxes).
cudaError_t launch_decompress(const CUtensorMap& tmC, const CUtensorMap& tmWK, const CUtensorMap& tmWV,
                              const int32_t* block_table, const int32_t* seq_lens, void* k_nope, void* v,
                              WsHeader* ws, int B, int H, int G, int Lq, int max_pages, int num_pages,
                              unsigned long long wait_ns, cudaStream_t st);
cudaError_t launch_prefill_attend(const CUtensorMap& tmQN, const CUtensorMap& tmQR, const CUtensorMap& tmK,
                                  const CUtensorMap& tmV, const CUtensorMap& tmC, const int32_t* block_table,
                                  const int32_t* seq_lens, void* out, float* lse, WsHeader* ws, int B, int Lq,
                                  int H, int max_pages, int num_pages, float scale, unsigned long long wait_ns,
                                  cudaStream_t st);
// CTAs per cluster of the decode launch: a pair per 128 query rows of a
// sequence (in solo mode each CTA of the pair holds half the heads)
inline bool decode_solo(int G) { return G > 1; }
inline int decode_plan_max_b(int G) { return decode_solo(G) ? kPlanInKernelMaxBSolo : kPlanInKernelMaxB; }
inline int decode_csize(int Lq, int H, int G) {
  const int rows_per_cta = decode_solo(G) ? Lq * (H / 2) : Lq * H;
  return 2 * ((rows_per_cta + kRowsPerCta - 1) / kRowsPerCta);
}

}  // namespace mla
