// mla_api.cu — the C ABI declared in include/mla.h: argument validation,
// tensor-map encoding, kernel launches.  No allocation, no global state
// beyond per-device launch-configuration caches and a cache of encoded
// tensor maps.
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "mla_internal.h"

using namespace mla;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encoded tensor maps, remembered by their complete encoding arguments: a
// decode step encodes about nine, and a serving loop passes the same
// buffers every step.  64 entries, replaced in turn; guarded by a mutex.
struct MapKey {
  const void* base;
  int rank, swz, type;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3];
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
constexpr int kMapCache = 64;
struct MapCache {
  uint64_t hash[kMapCache];  // scanned first; the key is compared only on a hash match
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int used = 0, next = 0;
};
// FNV-1a over the key's bytes
uint64_t map_hash(const MapKey& k) {
  const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
  return h;
}
std::mutex g_map_mu;
MapCache g_maps;

// Tensor map (bf16 and 128-byte swizzle unless told otherwise); dims
// innermost first; strides in bytes for dims 1..rank-1.
int make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
             const cuuint64_t* strides, const cuuint32_t* box,
             CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B,
             CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  if (rank < 1 || rank > 3) return MLA_ERR_INVALID_ARG;
  MapKey k;
  std::memset(&k, 0, sizeof(k));  // padding included: keys compare bytewise
  k.base = base;
  k.rank = rank;
  k.swz = (int)swz;
  k.type = (int)type;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  const uint64_t hk = map_hash(k);
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_maps.used; ++i)
      if (g_maps.hash[i] == hk && g_maps.key[i] == k) {
        *m = g_maps.map[i];
        return MLA_OK;
      }
  }
  auto fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = fn(m, type, rank, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_map_mu);
  const int slot = g_maps.used < kMapCache ? g_maps.used++ : (g_maps.next++ % kMapCache);
  g_maps.hash[slot] = hk;
  g_maps.key[slot] = k;
  g_maps.map[slot] = *m;
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const mla_dims* d) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->B < 1 || d->Lq < 1 || d->H < 1 || d->max_pages_per_seq < 1 || d->num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (!(d->scale > 0.f) || !std::isfinite(d->scale)) return MLA_ERR_INVALID_ARG;
  if (d->d_hc != kDhc || d->d_c != kDc || d->d_R != kDr || d->page_size != kPage)
    return MLA_ERR_UNSUPPORTED;
  if (d->G != 1 && d->G != 2 && d->G != 4 && d->G != 8) return MLA_ERR_UNSUPPORTED;
  if (d->Lq > 4 || d->H % 16 != 0 || d->H > 128 || d->H % d->G != 0) return MLA_ERR_UNSUPPORTED;
  // TMA row coordinate page*64 and table indices stay in int32
  if ((long long)d->num_pages * kPage >= (1LL << 31)) return MLA_ERR_UNSUPPORTED;
  if ((long long)d->B * d->max_pages_per_seq >= (1LL << 31)) return MLA_ERR_UNSUPPORTED;
  if ((long long)d->max_pages_per_seq * kPage >= (1LL << 31)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

// The decompress branch accepts any number of new tokens (up to the cached
// length); its tensor views index rows in int32.
int check_dims_prefill(const mla_dims* d) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->Lq < 1) return MLA_ERR_INVALID_ARG;
  mla_dims one = *d;
  one.Lq = 1;
  int rc = check_dims(&one);
  if (rc != MLA_OK) return rc;
  if (d->Lq > d->max_pages_per_seq * kPage) return MLA_ERR_INVALID_ARG;
  if ((long long)d->B * d->Lq >= (1LL << 31) || (long long)d->B * d->H * d->max_pages_per_seq * kPage >= (1LL << 31))
    return MLA_ERR_UNSUPPORTED;
  if (d->B > 65535) return MLA_ERR_UNSUPPORTED;  // grid z
  return MLA_OK;
}

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stall_page{-1};

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

int row_blocks(const mla_dims* d) { return (d->Lq * d->H + kRowsPerCta - 1) / kRowsPerCta; }

}  // namespace

namespace mla {
unsigned long long decode_wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int decode_stall_page() { return g_stall_page.load(std::memory_order_relaxed); }
int gemm_rows_box(int M);  // mla_gemm.cu: query rows per absorb/project CTA tile (the MMA's N)
}  // namespace mla

extern "C" {

int mla_set_timeout_test(long long wait_limit_ns, int stall_page) {
  if (wait_limit_ns < 0 || stall_page < -1) return MLA_ERR_INVALID_ARG;
  g_wait_ns.store(wait_limit_ns == 0 ? kDefaultWaitNs : (unsigned long long)wait_limit_ns,
                  std::memory_order_relaxed);
  g_stall_page.store(stall_page, std::memory_order_relaxed);
  return MLA_OK;
}

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_MISALIGNED: return "MLA_ERR_MISALIGNED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_BAD_TABLE: return "MLA_ERR_BAD_TABLE";
    case MLA_ERR_BAD_SEQLEN: return "MLA_ERR_BAD_SEQLEN";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_RANGE: return "MLA_ERR_RANGE";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_absorb_q(const mla_dims* d, const void* q_nope, const void* q_rope, const void* W_UK,
                 void* q_cat, void* stream) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!q_nope || !q_rope || !W_UK || !q_cat) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(W_UK) || !aligned16(q_cat))
    return MLA_ERR_MISALIGNED;
  const int M = d->B * d->Lq, H = d->H, dg = kDc / d->G;
  CUtensorMap tA, tB;
  {
    cuuint64_t dims[3] = {(cuuint64_t)kDhc, (cuuint64_t)H, (cuuint64_t)M};
    cuuint64_t strides[2] = {(cuuint64_t)kDhc * 2, (cuuint64_t)H * kDhc * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)gemm_rows_box(M)};
    if ((rc = make_map(&tA, q_nope, 3, dims, strides, box)) != MLA_OK) return rc;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)dg, (cuuint64_t)kDhc, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)dg * 2, (cuuint64_t)kDhc * dg * 2};
    cuuint32_t box[3] = {64, kDhc, 1};
    if ((rc = make_map(&tB, W_UK, 3, dims, strides, box)) != MLA_OK) return rc;
  }
  return cuda_status(launch_absorb(tA, tB, q_rope, q_cat, M, H, dg, static_cast<cudaStream_t>(stream)));
}

int mla_project_uv(const mla_dims* d, const void* o_lat, const void* W_UV, void* out, void* stream) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!o_lat || !W_UV || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(W_UV) || !aligned16(out)) return MLA_ERR_MISALIGNED;
  const int M = d->B * d->Lq, H = d->H, dg = kDc / d->G;
  CUtensorMap tA, tB;
  {
    cuuint64_t dims[3] = {(cuuint64_t)dg, (cuuint64_t)H, (cuuint64_t)M};
    cuuint64_t strides[2] = {(cuuint64_t)dg * 2, (cuuint64_t)H * dg * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)gemm_rows_box(M)};
    if ((rc = make_map(&tA, o_lat, 3, dims, strides, box)) != MLA_OK) return rc;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)dg, (cuuint64_t)kDhc, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)dg * 2, (cuuint64_t)kDhc * dg * 2};
    cuuint32_t box[3] = {64, kDhc, 1};  // all 128 output rows of W_UV[h] per CTA
    if ((rc = make_map(&tB, W_UV, 3, dims, strides, box)) != MLA_OK) return rc;
  }
  return cuda_status(launch_project(tA, tB, out, M, H, dg, static_cast<cudaStream_t>(stream)));
}

int mla_decode_workspace_size(const mla_dims* d, size_t* bytes) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!bytes) return MLA_ERR_INVALID_ARG;
  *bytes = ws_bytes_for(d->B);
  return MLA_OK;
}

int mla_decode_num_slots(const mla_dims* d, int* slots) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!slots) return MLA_ERR_INVALID_ARG;
  int units = 0;
  if ((rc = decode_max_units(decode_solo(d->G), false, decode_csize(d->Lq, d->H, d->G), &units)) != MLA_OK)
    return rc;
  *slots = d->B + units - 1;
  return MLA_OK;
}

int mla_decode_kernel_launches(const mla_dims* d, int* launches) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!launches) return MLA_ERR_INVALID_ARG;
  *launches = d->B <= decode_plan_max_b(d->G) ? 1 : 2;
  return MLA_OK;
}

}  // extern "C"

namespace {
// mla_decode_paged and mla_decode_paged_fp8: the same kernel, with the
// cache rows in bf16 or FP8.
int decode_paged(const mla_dims* d, const void* q_cat, const void* kv_cache, bool fp8,
                 const int32_t* block_table, const int32_t* seq_lens, int num_splits, float* o_part,
                 float* lse_part, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!q_cat || !kv_cache || !block_table || !seq_lens || !o_part || !lse_part || num_splits < 0)
    return MLA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < ws_bytes_for(d->B)) return MLA_ERR_WORKSPACE;
  if (!aligned16(q_cat) || !aligned16(kv_cache) || !aligned16(o_part) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse_part) & 3u))
    return MLA_ERR_MISALIGNED;
  const bool solo = decode_solo(d->G);
  const int csize = decode_csize(d->Lq, d->H, d->G);
  int units = 0;
  if ((rc = decode_max_units(solo, false, csize, &units)) != MLA_OK) return rc;
  if (fp8) {  // never more units than mla_decode_num_slots counts on
    int units8 = 0;
    if ((rc = decode_max_units(solo, true, csize, &units8)) != MLA_OK) return rc;
    if (units8 < units) units = units8;
  }
  if (num_splits > 0 && num_splits < units) units = num_splits;
  auto st = static_cast<cudaStream_t>(stream);
  CUtensorMap tm, tm_rope, tm_qrope, tm_qlat, tm_scale;
  const cuuint64_t rows = (cuuint64_t)d->num_pages * kPage;
  if (fp8) {
    // the same rows seen as bytes (codes), bf16 (RoPE key) and fp32 (scales)
    const cuuint64_t strides[1] = {(cuuint64_t)kRowBytesFp8};
    const cuuint64_t dims8[2] = {(cuuint64_t)kRowBytesFp8, rows};
    const cuuint32_t box8[2] = {64, kPage};
    if ((rc = make_map(&tm, kv_cache, 2, dims8, strides, box8, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_DATA_TYPE_UINT8)) != MLA_OK)
      return rc;
    const cuuint64_t dims16[2] = {(cuuint64_t)kRowBytesFp8 / 2, rows};
    const cuuint32_t rbox[2] = {32, kPage};
    if ((rc = make_map(&tm_rope, kv_cache, 2, dims16, strides, rbox, CU_TENSOR_MAP_SWIZZLE_64B)) != MLA_OK)
      return rc;
    const cuuint64_t dims32[2] = {(cuuint64_t)kRowBytesFp8 / 4, rows};
    const cuuint32_t sbox[2] = {4, kPage};
    if ((rc = make_map(&tm_scale, kv_cache, 2, dims32, strides, sbox, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) != MLA_OK)
      return rc;
  } else {
    cuuint64_t dims[2] = {(cuuint64_t)kRow, rows};
    cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
    cuuint32_t box[2] = {64, kPage};
    if ((rc = make_map(&tm, kv_cache, 2, dims, strides, box)) != MLA_OK) return rc;
    cuuint32_t rbox[2] = {32, kPage};
    if ((rc = make_map(&tm_rope, kv_cache, 2, dims, strides, rbox, CU_TENSOR_MAP_SWIZZLE_64B)) != MLA_OK)
      return rc;
    tm_scale = tm;  // not read
  }
  {
    const int d_q = kDc / d->G + kDr;
    cuuint64_t dims[2] = {(cuuint64_t)d_q, (cuuint64_t)d->B * d->Lq * d->H};
    cuuint64_t strides[1] = {(cuuint64_t)d_q * 2};
    // RoPE query boxes: 128 rows (pair mode) or the H/2 heads of one token (solo mode)
    cuuint32_t box[2] = {32, solo ? (cuuint32_t)(d->H / 2) : (cuuint32_t)kRowsPerCta};
    if ((rc = make_map(&tm_qrope, q_cat, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B)) != MLA_OK) return rc;
    cuuint32_t lbox[2] = {64, kRowsPerCta};
    if ((rc = make_map(&tm_qlat, q_cat, 2, dims, strides, lbox)) != MLA_OK) return rc;
  }
  auto* ws = static_cast<WsHeader*>(workspace);
  // Small batches are split by the decode kernel itself (one launch);
  // larger ones by the separate plan kernel.
  const bool in_kernel = d->B <= decode_plan_max_b(d->G);
  if (!in_kernel) {
    cudaError_t e = launch_plan(seq_lens, block_table, ws, d->B, d->Lq, d->max_pages_per_seq,
                                d->num_pages, units, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
  }
  DecodeArgs a;
  a.q_cat = static_cast<const __nv_bfloat16*>(q_cat);
  a.block_table = block_table;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.ws = ws;
  a.B = d->B;
  a.Lq = d->Lq;
  a.H = d->H;
  a.G = d->G;
  a.d_g = kDc / d->G;
  a.max_pages = d->max_pages_per_seq;
  a.num_pages = d->num_pages;
  a.causal = d->causal ? 1 : 0;
  a.rows = d->Lq * d->H;
  a.scale_log2 = d->scale * 1.4426950408889634f;
  a.plan_in_kernel = in_kernel ? 1 : 0;
  a.units = units;
  a.seq_lens = seq_lens;
  a.wait_ns = decode_wait_limit_ns();
  a.stall_page = decode_stall_page();
  return cuda_status(launch_decode(solo, fp8, tm, tm_rope, tm_qrope, tm_qlat, tm_scale, a, units, csize, st));
}
}  // namespace

extern "C" {

int mla_decode_paged(const mla_dims* d, const void* q_cat, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens, int num_splits,
                     float* o_part, float* lse_part, void* workspace, size_t ws_bytes, void* stream) {
  return decode_paged(d, q_cat, kv_cache, false, block_table, seq_lens, num_splits, o_part, lse_part, workspace,
                      ws_bytes, stream);
}

int mla_decode_paged_fp8(const mla_dims* d, const void* q_cat, const void* kv_cache_fp8,
                         const int32_t* block_table, const int32_t* seq_lens, int num_splits,
                         float* o_part, float* lse_part, void* workspace, size_t ws_bytes, void* stream) {
  return decode_paged(d, q_cat, kv_cache_fp8, true, block_table, seq_lens, num_splits, o_part, lse_part, workspace,
                      ws_bytes, stream);
}

int mla_combine_splits(const mla_dims* d, const float* o_part, const float* lse_part,
                       const void* workspace, size_t ws_bytes, void* o_lat, float* lse,
                       void* stream) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!o_part || !lse_part || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < ws_bytes_for(d->B)) return MLA_ERR_WORKSPACE;
  if (!aligned16(o_part) || !aligned16(o_lat) || !aligned16(workspace)) return MLA_ERR_MISALIGNED;
  int slots = 0;
  if ((rc = mla_decode_num_slots(d, &slots)) != MLA_OK) return rc;
  return cuda_status(launch_combine(o_part, lse_part, static_cast<const WsHeader*>(workspace), o_lat,
                                    lse, d->B, d->Lq, d->H, d->G, slots, static_cast<cudaStream_t>(stream)));
}

int mla_combine_project(const mla_dims* d, const float* o_part, const float* lse_part, const void* workspace,
                        size_t ws_bytes, const void* W_UV, void* out, void* o_lat, float* lse, void* stream) {
  int rc = check_dims(d);
  if (rc != MLA_OK) return rc;
  if (!o_part || !lse_part || !W_UV || !out) return MLA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < ws_bytes_for(d->B)) return MLA_ERR_WORKSPACE;
  if (!aligned16(o_part) || !aligned16(W_UV) || !aligned16(out) || !aligned16(workspace) ||
      (o_lat && !aligned16(o_lat)) || (reinterpret_cast<uintptr_t>(lse_part) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_MISALIGNED;
  const int H = d->H, dg = kDc / d->G;
  CUtensorMap tA;
  {
    cuuint64_t dims[3] = {(cuuint64_t)dg, (cuuint64_t)kDhc, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)dg * 2, (cuuint64_t)kDhc * dg * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kDhc, 1};  // all 128 output rows of W_UV[h], 64 latent columns
    if ((rc = make_map(&tA, W_UV, 3, dims, strides, box)) != MLA_OK) return rc;
  }
  int slots = 0;
  if ((rc = mla_decode_num_slots(d, &slots)) != MLA_OK) return rc;
  return cuda_status(launch_combine_project(tA, o_part, lse_part, static_cast<const WsHeader*>(workspace), out,
                                            o_lat, lse, d->B, d->Lq, d->H, d->G, slots,
                                            static_cast<cudaStream_t>(stream)));
}

int mla_decompressed_kv_size(const mla_dims* d, size_t* bytes) {
  int rc = check_dims_prefill(d);
  if (rc != MLA_OK) return rc;
  if (!bytes) return MLA_ERR_INVALID_ARG;
  *bytes = (size_t)d->B * d->H * d->max_pages_per_seq * kPage * kDhc * 2;
  return MLA_OK;
}

int mla_decompress_kv(const mla_dims* d, const void* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, const void* W_UK, const void* W_UV, void* k_nope, void* v,
                      void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_dims_prefill(d);
  if (rc != MLA_OK) return rc;
  if (!kv_cache || !block_table || !seq_lens || !W_UK || !W_UV || !k_nope || !v) return MLA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < sizeof(WsHeader)) return MLA_ERR_WORKSPACE;
  if (!aligned16(kv_cache) || !aligned16(W_UK) || !aligned16(W_UV) || !aligned16(k_nope) || !aligned16(v) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 3u))
    return MLA_ERR_MISALIGNED;
  const int H = d->H, dg = kDc / d->G;
  CUtensorMap tC, tK, tV;
  {
    cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)d->num_pages * kPage};
    cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
    cuuint32_t box[2] = {64, kPage};
    if ((rc = make_map(&tC, kv_cache, 2, dims, strides, box)) != MLA_OK) return rc;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)dg, (cuuint64_t)kDhc, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)dg * 2, (cuuint64_t)kDhc * dg * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kDhc, 1};
    if ((rc = make_map(&tK, W_UK, 3, dims, strides, box)) != MLA_OK) return rc;
    if ((rc = make_map(&tV, W_UV, 3, dims, strides, box)) != MLA_OK) return rc;
  }
  return cuda_status(launch_decompress(tC, tK, tV, block_table, seq_lens, k_nope, v,
                                       static_cast<WsHeader*>(workspace), d->B, H, d->G, d->Lq,
                                       d->max_pages_per_seq, d->num_pages, decode_wait_limit_ns(),
                                       static_cast<cudaStream_t>(stream)));
}

int mla_prefill_attend(const mla_dims* d, const void* q_nope, const void* q_rope, const void* kv_cache,
                       const int32_t* block_table, const int32_t* seq_lens, const void* k_nope, const void* v,
                       void* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_dims_prefill(d);
  if (rc != MLA_OK) return rc;
  if (!q_nope || !q_rope || !kv_cache || !block_table || !seq_lens || !k_nope || !v || !out || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < sizeof(WsHeader)) return MLA_ERR_WORKSPACE;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(kv_cache) || !aligned16(k_nope) || !aligned16(v) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 3u))
    return MLA_ERR_MISALIGNED;
  const int H = d->H;
  const cuuint64_t rows_q = (cuuint64_t)d->B * d->Lq, rows_kv = (cuuint64_t)d->B * H * d->max_pages_per_seq * kPage;
  CUtensorMap tQN, tQR, tK, tV, tC;
  {
    cuuint64_t dims[2] = {(cuuint64_t)H * kDhc, rows_q};
    cuuint64_t strides[1] = {(cuuint64_t)H * kDhc * 2};
    cuuint32_t box[2] = {64, kRowsPerCta};
    if ((rc = make_map(&tQN, q_nope, 2, dims, strides, box)) != MLA_OK) return rc;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)H * kDr, rows_q};
    cuuint64_t strides[1] = {(cuuint64_t)H * kDr * 2};
    cuuint32_t box[2] = {64, kRowsPerCta};
    if ((rc = make_map(&tQR, q_rope, 2, dims, strides, box)) != MLA_OK) return rc;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)kDhc, rows_kv};
    cuuint64_t strides[1] = {(cuuint64_t)kDhc * 2};
    cuuint32_t box[2] = {64, kPage};
    if ((rc = make_map(&tK, k_nope, 2, dims, strides, box)) != MLA_OK) return rc;
    if ((rc = make_map(&tV, v, 2, dims, strides, box)) != MLA_OK) return rc;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)d->num_pages * kPage};
    cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
    cuuint32_t box[2] = {64, kPage};
    if ((rc = make_map(&tC, kv_cache, 2, dims, strides, box)) != MLA_OK) return rc;
  }
  return cuda_status(launch_prefill_attend(tQN, tQR, tK, tV, tC, block_table, seq_lens, out, lse,
                                           static_cast<WsHeader*>(workspace), d->B, d->Lq, H,
                                           d->max_pages_per_seq, d->num_pages, d->scale, decode_wait_limit_ns(),
                                           static_cast<cudaStream_t>(stream)));
}

int mla_decode_step(const mla_dims* d, const void* q_nope, const void* q_rope, const void* W_UK, const void* W_UV,
                    const void* kv_cache, int kv_fp8, const int32_t* block_table, const int32_t* seq_lens,
                    void* q_cat, float* o_part, float* lse_part, void* workspace, size_t ws_bytes, void* o_lat,
                    float* lse, void* out, int fused, void* stream) {
  if (!out) return MLA_ERR_INVALID_ARG;
  if (!fused && !o_lat) return MLA_ERR_INVALID_ARG;
  int rc = mla_absorb_q(d, q_nope, q_rope, W_UK, q_cat, stream);
  if (rc != MLA_OK) return rc;
  rc = kv_fp8 ? mla_decode_paged_fp8(d, q_cat, kv_cache, block_table, seq_lens, 0, o_part, lse_part, workspace,
                                     ws_bytes, stream)
              : mla_decode_paged(d, q_cat, kv_cache, block_table, seq_lens, 0, o_part, lse_part, workspace, ws_bytes,
                                 stream);
  if (rc != MLA_OK) return rc;
  if (fused) return mla_combine_project(d, o_part, lse_part, workspace, ws_bytes, W_UV, out, o_lat, lse, stream);
  rc = mla_combine_splits(d, o_part, lse_part, workspace, ws_bytes, o_lat, lse, stream);
  if (rc != MLA_OK) return rc;
  return mla_project_uv(d, o_lat, W_UV, out, stream);
}

int mla_get_device_status(const void* workspace, void* stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  int status = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  return status;
}

}  // extern "C"
