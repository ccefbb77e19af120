// C ABI of libfa.so (declared in include/fa.h): argument checks, tensor-map
// encoding, grid sizing and dispatch to the (D, causal) kernel instantiations.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "../../include/fa.h"
#include "fa_kernels.h"
#include "tma_host.h"

// The library's only device state: one status word per device (0 = ok).
__device__ int g_fa_status = 0;

#include "ptx.cuh"

// Waits on a barrier that is never signalled: exercises the bounded wait,
// the status report and the clean exit of a kernel that gave up.
__global__ void fa_selftest_wait_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(&bar, 1);
    abort_flag = 0;
    fa::fence_barrier_init();
  }
  __syncthreads();
  const fa::WaitCtx wc{status, &abort_flag};
  if (threadIdx.x == 0) fa::mbar_wait(&bar, 0, wc, 200);
  __syncthreads();
}

namespace {

struct DevInfo {
  bool init = false;
  int sms = 0;
  int* status = nullptr;  // device address of g_fa_status on this device
};

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];

int current_device_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    if (major != 10 || minor != 3) return FA_ERR_DEVICE;
    if (const char* env = std::getenv("FA_NUM_SMS")) {
      const int v = std::atoi(env);
      if (v > 0 && v < sms) sms = v;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
    d.sms = sms;
    d.status = static_cast<int*>(p);
    d.init = true;
  }
  *out = &d;
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Problem shape of one call: queries [Z, H, Nq, D], keys/values [Z, Hkv, Nk, D].
struct Shape {
  int Z, H, Hkv, Nq, Nk, D;
  int causal;
  long long q_heads() const { return static_cast<long long>(Z) * H; }
  long long kv_heads() const { return static_cast<long long>(Z) * Hkv; }
  int group() const { return H / Hkv; }
  int nq_pad() const { return (Nq + 127) / 128 * 128; }
};

// Shared checks of the shape arguments.
int check_shape(const Shape& sh, float scale) {
  if (sh.Z <= 0 || sh.H <= 0 || sh.Hkv <= 0 || sh.Nq <= 0 || sh.Nk <= 0) return FA_ERR_INVALID_ARG;
  if (sh.H % sh.Hkv != 0) return FA_ERR_INVALID_ARG;
  if (sh.causal != 0 && sh.causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (sh.D != 64 && sh.D != 128 && sh.D != 256) return FA_ERR_UNSUPPORTED;
  // causal with more queries than keys leaves rows with no visible key
  if (sh.causal && sh.Nq > sh.Nk) return FA_ERR_UNSUPPORTED;
  // 32-bit row and element-offset arithmetic inside the kernels
  if (sh.q_heads() * sh.nq_pad() >= (1LL << 31) || sh.kv_heads() * sh.Nk >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

Shape square(int Z, int H, int N, int D, int causal) { return Shape{Z, H, H, N, N, D, causal}; }

// `mats` matrices [rows x D] of 16-bit elements (fp16, or bf16 when
// `bf16`), one after the other; boxes of 64 columns x box_rows rows.
bool map16(CUtensorMap* m, const void* base, long long mats, int rows, int D, int box_rows, bool bf16) {
  std::memset(m, 0, sizeof(*m));
  return fa::make_tmap_3d(m, base, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          static_cast<uint64_t>(mats), static_cast<uint64_t>(rows), static_cast<uint64_t>(D), 64,
                          static_cast<uint32_t>(box_rows), true);
}

constexpr float kLog2e = 1.4426950408889634f;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout of fa_bwd: [delta | lse2], each [Z*H, Nq_pad] fp32 (query
// rows padded to whole 128-row tiles) and 256-byte aligned.  Nothing else:
// every dQ, dK and dV tile is accumulated on chip by the CTA that owns it.
struct BwdWorkspace {
  size_t delta_off, lse2_off, total;
};

BwdWorkspace bwd_workspace_layout(const Shape& sh) {
  BwdWorkspace w{};
  const size_t vec = round_up(static_cast<size_t>(sh.q_heads()) * sh.nq_pad() * sizeof(float), 256);
  w.delta_off = 0;
  w.lse2_off = vec;
  w.total = 2 * vec;
  return w;
}

}  // namespace

extern "C" {

const char* fa_error_string(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, non-positive size, bad scale or causal flag)";
    case FA_ERR_UNSUPPORTED: return "unsupported shape (D must be 64, 128 or 256; causal needs Nq <= Nk; Z*H*N < 2^31)";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than its size query returns";
    case FA_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case FA_ERR_DEVICE: return "current device is not a compute capability 10.3 (sm_103a) GPU";
    case FA_ERR_TIMEOUT: return "a device-side wait gave up; outputs since the last status check are invalid";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than fa_bwd_noalloc's built-in 64 MiB buffer";
    default: return "unknown error code";
  }
}

long long fa_fwd_tile_count(int N, int D, int causal) {
  if (N <= 0 || (D != 64 && D != 128 && D != 256) || (causal != 0 && causal != 1)) return -1;
  const long long bm = 128, bn = fa::fwd_dense_block_n(D);
  const long long nqt = (N + bm - 1) / bm, nkv = (N + bn - 1) / bn;
  if (!causal) return nqt * nkv;
  long long n = 0;
  for (long long qt = 0; qt < nqt; ++qt) {
    const long long end = (qt + 1) * bm < N ? (qt + 1) * bm : N;  // one past the tile's last visible key
    n += (end + bn - 1) / bn;
  }
  return n;
}

double fa_fwd_ex_flops(int Z, int H, int Nq, int Nk, int D, int causal) {
  const double heads = static_cast<double>(Z) * H, nq = Nq, d = D;
  // (query, key) pairs that take part: all, or query i sees i + Nk - Nq + 1 keys
  const double pairs = causal ? nq * (nq + 1.0) / 2.0 + nq * (static_cast<double>(Nk) - Nq) : nq * Nk;
  return heads * 4.0 * pairs * d;
}

double fa_fwd_flops(int Z, int H, int N, int D, int causal) { return fa_fwd_ex_flops(Z, H, N, N, D, causal); }

double fa_bwd_flops(int Z, int H, int N, int D, int causal) { return 2.5 * fa_fwd_flops(Z, H, N, D, causal); }

double fa_bwd_ex_flops(int Z, int H, int Nq, int Nk, int D, int causal) {
  return 2.5 * fa_fwd_ex_flops(Z, H, Nq, Nk, D, causal);
}

}  // extern "C"

namespace {

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const Shape& sh, float scale,
             cudaStream_t stream, bool bf16) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  int rc = check_shape(sh, scale);
  if (rc != FA_OK) return rc;
  DevInfo* dev = nullptr;
  if ((rc = current_device_info(&dev)) != FA_OK) return rc;

  const int D = sh.D;
  const int bn = fa::fwd_dense_block_n(D);
  const int bv = D == 256 ? 64 : bn;  // D = 256: V in halves of the keys
  // Few queries per head (decode): the G query heads of a K/V head run as one
  // head of G * Nq rows (consecutive in q, o and lse), so K/V tiles are read
  // once per K/V head and the 128-row query tiles are filled.
  const bool pack = sh.group() > 1 && sh.group() * sh.Nq <= 128;
  const long long qh = pack ? sh.kv_heads() : sh.q_heads();
  const int rows = pack ? sh.group() * sh.Nq : sh.Nq;
  CUtensorMap maps[4];  // q, k, v, o
  if (!map16(&maps[0], q, qh, rows, D, 128, bf16) || !map16(&maps[1], k, sh.kv_heads(), sh.Nk, D, bn, bf16) ||
      !map16(&maps[2], v, sh.kv_heads(), sh.Nk, D, bv, bf16) || !map16(&maps[3], o, qh, rows, D, 128, bf16))
    return FA_ERR_CUDA;
  fa::FwdParams prm{};
  prm.o = static_cast<__half*>(o);
  prm.lse = lse;
  prm.heads = static_cast<int>(qh);
  prm.group = pack ? 1 : sh.group();
  prm.q_period = pack ? sh.Nq : 0;
  prm.Nq = rows;
  prm.Nk = sh.Nk;
  prm.causal_off = sh.Nk - sh.Nq;
  prm.scale_log2 = scale * kLog2e;
  prm.status = dev->status;
  const bool c = sh.causal != 0;
  switch (D) {
    case 64: rc = fa::launch_fwd_d64(c, bf16, maps, prm, dev->sms, stream); break;
    case 128: rc = fa::launch_fwd_d128(c, bf16, maps, prm, dev->sms, stream); break;
    default: rc = fa::launch_fwd_d256(c, bf16, maps, prm, dev->sms, stream); break;
  }
  return rc == 0 ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int H, int N, int D,
           int causal, float scale, cudaStream_t stream) {
  return fwd_impl(q, k, v, o, lse, square(Z, H, N, D, causal), scale, stream, false);
}

int fa_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int H, int N, int D,
                int causal, float scale, cudaStream_t stream) {
  return fwd_impl(q, k, v, o, lse, square(Z, H, N, D, causal), scale, stream, true);
}

int fa_reshape_and_cache(const void* k_new, const void* v_new, const long long* slot_mapping, void* k_cache,
                         void* v_cache, int tokens, int Hkv, int D, int num_pages, int page_size,
                         cudaStream_t stream) {
  if (tokens < 0 || Hkv <= 0 || D <= 0 || num_pages <= 0 || page_size <= 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (tokens == 0) return FA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return FA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return FA_ERR_INVALID_ARG;
  DevInfo* dev = nullptr;
  const int rc = current_device_info(&dev);
  if (rc != FA_OK) return rc;
  const long long rows = static_cast<long long>(num_pages) * page_size;
  return fa::launch_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, tokens, Hkv, D, rows, dev->sms,
                                stream) == 0
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Split paged forward workspace: per-slice lse [splits, rows] then per-slice
// O [splits, rows, D], fp32, rows = B * H * Nq (query rows of the call).
constexpr int kMaxSplits = 256;
long long split_lse_bytes(long long rows, int splits) { return (rows * splits * 4 + 255) / 256 * 256; }
long long split_workspace_bytes(long long rows, int D, int splits) {
  return split_lse_bytes(rows, splits) + rows * splits * D * 4;
}

// Shared by the paged, the split paged and the selected-block forward:
// argument checks, the 4-D cache maps and the launch.  `lists` is the block
// table (paged) or the selected-page list (sparse); `blocks` and `counts` are
// the sparse-only logical blocks and selection counts; `splits` and the
// workspace are the split mode's (mode 3).
int paged_impl(int mode, const void* q, const void* k_cache, const void* v_cache, const int* lists,
               const int* blocks, const int* counts, const int* context_lens, void* o, float* lse, int B, int H,
               int Hkv, int Nq, int D, int num_pages, int page_size, int max_entries, int causal, float scale,
               int dtype, int splits, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const bool sparse = mode == 2, split = mode == 3;
  if (split && (splits < 1 || splits > kMaxSplits)) return FA_ERR_INVALID_ARG;
  if (split && (!workspace || !aligned(workspace, 16))) return FA_ERR_WORKSPACE;
  if (!q || !k_cache || !v_cache || !lists || !context_lens || !o || !lse) return FA_ERR_INVALID_ARG;
  if (sparse && (!blocks || !counts)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(lists, 4) || !aligned(context_lens, 4) || (sparse && (!aligned(blocks, 4) || !aligned(counts, 4))))
    return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Hkv <= 0 || Nq <= 0 || num_pages <= 0 || page_size <= 0 || max_entries <= 0)
    return FA_ERR_INVALID_ARG;
  if (H % Hkv != 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  // a key tile is a whole number of pages, each a whole number of 8-row swizzle atoms
  if ((page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) || page_size > fa::fwd_block_n(D))
    return FA_ERR_UNSUPPORTED;
  const long long nq_pad = (Nq + 127LL) / 128 * 128;
  if (static_cast<long long>(B) * H * nq_pad >= (1LL << 31) ||
      static_cast<long long>(max_entries) * page_size >= (1LL << 31) ||
      static_cast<long long>(B) * (sparse ? Hkv : 1) * max_entries >= (1LL << 31))
    return FA_ERR_UNSUPPORTED;
  DevInfo* dev = nullptr;
  int rc = current_device_info(&dev);
  if (rc != FA_OK) return rc;
  const bool bf16 = dtype == FA_DTYPE_BF16;
  const auto et = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // decode-sized calls pack the query heads of a K/V head (see fwd_impl)
  const int g = H / Hkv;
  const bool pack = g > 1 && g * Nq <= 128;
  const int hps = pack ? Hkv : H;         // (packed) query heads per sequence
  const int rows = pack ? g * Nq : Nq;
  CUtensorMap maps[4];  // q, k cache, v cache, o
  std::memset(&maps[1], 0, sizeof(CUtensorMap));
  std::memset(&maps[2], 0, sizeof(CUtensorMap));
  if (!map16(&maps[0], q, static_cast<long long>(B) * hps, rows, D, 128, bf16) ||
      !fa::make_tmap_paged(&maps[1], k_cache, et, 2, num_pages, page_size, Hkv, D, 64, true) ||
      !fa::make_tmap_paged(&maps[2], v_cache, et, 2, num_pages, page_size, Hkv, D, 64, true) ||
      !map16(&maps[3], o, static_cast<long long>(B) * hps, rows, D, 128, bf16))
    return FA_ERR_CUDA;
  fa::FwdParams prm{};
  prm.o = static_cast<__half*>(o);
  prm.lse = lse;
  prm.heads = B * hps;
  prm.group = pack ? 1 : g;
  prm.q_period = pack ? Nq : 0;
  prm.Nq = rows;
  prm.Nk = max_entries * page_size;  // per sequence: context_lens[b] (paged), the selection (sparse)
  prm.causal_off = 0;
  prm.scale_log2 = scale * kLog2e;
  prm.status = dev->status;
  prm.block_table = sparse ? nullptr : lists;
  prm.sel_pages = sparse ? lists : nullptr;
  prm.sel_blocks = blocks;
  prm.sel_count = counts;
  prm.context_lens = context_lens;
  prm.H = hps;
  prm.Hkv = Hkv;
  prm.num_pages = num_pages;
  prm.page_size = page_size;
  prm.max_pages = max_entries;
  prm.splits = 1;
  if (split) {
    const long long rows_total = static_cast<long long>(B) * H * Nq;
    if (static_cast<unsigned long long>(split_workspace_bytes(rows_total, D, splits)) > workspace_bytes)
      return FA_ERR_WORKSPACE;
    prm.splits = splits;
    prm.part_lse = static_cast<float*>(workspace);
    prm.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + split_lse_bytes(rows_total, splits));
  }
  const bool c = causal != 0;
  if (split) {
    switch (D) {
      case 64: rc = fa::launch_fwd_paged_split_d64(c, bf16, maps, prm, dev->sms, stream); break;
      case 128: rc = fa::launch_fwd_paged_split_d128(c, bf16, maps, prm, dev->sms, stream); break;
      default: rc = fa::launch_fwd_paged_split_d256(c, bf16, maps, prm, dev->sms, stream); break;
    }
  } else if (sparse) {
    switch (D) {
      case 64: rc = fa::launch_fwd_sparse_d64(c, bf16, maps, prm, dev->sms, stream); break;
      case 128: rc = fa::launch_fwd_sparse_d128(c, bf16, maps, prm, dev->sms, stream); break;
      default: rc = fa::launch_fwd_sparse_d256(c, bf16, maps, prm, dev->sms, stream); break;
    }
  } else {
    switch (D) {
      case 64: rc = fa::launch_fwd_paged_d64(c, bf16, maps, prm, dev->sms, stream); break;
      case 128: rc = fa::launch_fwd_paged_d128(c, bf16, maps, prm, dev->sms, stream); break;
      default: rc = fa::launch_fwd_paged_d256(c, bf16, maps, prm, dev->sms, stream); break;
    }
  }
  return rc == 0 ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                 const int* context_lens, void* o, float* lse, int B, int H, int Hkv, int Nq, int D, int num_pages,
                 int page_size, int max_pages, int causal, float scale, int dtype, cudaStream_t stream) {
  return paged_impl(1, q, k_cache, v_cache, block_table, nullptr, nullptr, context_lens, o, lse, B, H, Hkv, Nq, D,
                    num_pages, page_size, max_pages, causal, scale, dtype, 1, nullptr, 0, stream);
}

size_t fa_fwd_paged_split_workspace_size(int B, int H, int Nq, int D, int num_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || num_splits < 1 || num_splits > kMaxSplits) return 0;
  if (D != 64 && D != 128 && D != 256) return 0;
  return split_workspace_bytes(static_cast<long long>(B) * H * Nq, D, num_splits);
}

int fa_fwd_paged_split_count(int B, int H, int Hkv, int Nq, int D, int page_size, int max_pages, int causal) {
  if (B <= 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || Nq <= 0 || page_size <= 0 || max_pages <= 0) return 1;
  if (D != 64 && D != 128 && D != 256) return 1;
  DevInfo* dev = nullptr;
  if (current_device_info(&dev) != FA_OK) return 1;
  const int g = H / Hkv;
  const bool pack = g > 1 && g * Nq <= 128;
  const long long rows = pack ? static_cast<long long>(g) * Nq : Nq;
  const long long nqt = (rows + 127) / 128;
  const long long per_head = causal ? (nqt + 1) / 2 : nqt;
  const long long units = static_cast<long long>(B) * (pack ? Hkv : H) * per_head;
  const long long tiles = (static_cast<long long>(max_pages) * page_size + fa::fwd_block_n(D) - 1) / fa::fwd_block_n(D);
  // one wave: as many slices as keep every unit on its own SM, never more
  // slices than key tiles
  long long s = units >= dev->sms ? 1 : dev->sms / units;
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  return static_cast<int>(s < 1 ? 1 : s);
}

int fa_fwd_paged_split(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                       const int* context_lens, void* o, float* lse, void* workspace, size_t workspace_bytes, int B,
                       int H, int Hkv, int Nq, int D, int num_pages, int page_size, int max_pages, int num_splits,
                       int causal, float scale, int dtype, cudaStream_t stream) {
  if (num_splits == 1)
    return paged_impl(1, q, k_cache, v_cache, block_table, nullptr, nullptr, context_lens, o, lse, B, H, Hkv, Nq,
                      D, num_pages, page_size, max_pages, causal, scale, dtype, 1, nullptr, 0, stream);
  return paged_impl(3, q, k_cache, v_cache, block_table, nullptr, nullptr, context_lens, o, lse, B, H, Hkv, Nq, D,
                    num_pages, page_size, max_pages, causal, scale, dtype, num_splits, workspace, workspace_bytes,
                    stream);
}

int fa_fwd_sparse(const void* q, const void* k_cache, const void* v_cache, const int* sel_pages,
                  const int* sel_blocks, const int* sel_count, const int* context_lens, void* o, float* lse, int B,
                  int H, int Hkv, int Nq, int D, int num_pages, int page_size, int max_sel, int causal, float scale,
                  int dtype, cudaStream_t stream) {
  return paged_impl(2, q, k_cache, v_cache, sel_pages, sel_blocks, sel_count, context_lens, o, lse, B, H, Hkv, Nq,
                    D, num_pages, page_size, max_sel, causal, scale, dtype, 1, nullptr, 0, stream);
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int H, int Hkv, int Nq,
              int Nk, int D, int causal, float scale, int dtype, cudaStream_t stream) {
  if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, Shape{Z, H, Hkv, Nq, Nk, D, causal}, scale, stream, dtype == FA_DTYPE_BF16);
}

size_t fa_bwd_ex_workspace_size(int Z, int H, int Hkv, int Nq, int Nk, int D, int causal) {
  const Shape sh{Z, H, Hkv, Nq, Nk, D, causal};
  if (check_shape(sh, 1.f) != FA_OK) return 0;
  return bwd_workspace_layout(sh).total;
}

size_t fa_bwd_workspace_size(int Z, int H, int N, int D, int causal) {
  return fa_bwd_ex_workspace_size(Z, H, H, N, N, D, causal);
}

}  // extern "C"

namespace {

// Argument checks shared by every backward entry point.
int bwd_checks(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               const void* dq, const void* dk, const void* dv, const Shape& sh, float scale) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  return check_shape(sh, scale);
}

// Tensor maps of a backward call (box rows chosen by the kernels' tiling):
// [0] q, [1] k, [2] v, [3] dout, then the outputs [4] dq, [5] dk, [6] dv
// (TMA stores of the D <= 128 kernels); for D = 256, [0] and [3] have the
// dK/dV kernel's 64-row query tiles and [7] q, [8] k, [2] v the dQ kernel's
// 128-row query tiles and 64-row key tiles; [9] the forward output o
// (128-row tiles, read by the D <= 128 dQ kernel to form Delta).
constexpr int kBwdMaps = 10;
bool bwd_maps(CUtensorMap* maps, const void* q, const void* k, const void* v, const void* o, const void* dout,
              void* dq, void* dk, void* dv, const Shape& sh, bool bf16) {
  const int D = sh.D;
  const int bq = (D == 256) ? 64 : 128, bv = (D == 256) ? 64 : 128;
  const long long hq = sh.q_heads(), hk = sh.kv_heads();
  return map16(&maps[0], q, hq, sh.Nq, D, bq, bf16) && map16(&maps[1], k, hk, sh.Nk, D, 128, bf16) &&
         map16(&maps[2], v, hk, sh.Nk, D, bv, bf16) && map16(&maps[3], dout, hq, sh.Nq, D, bq, bf16) &&
         map16(&maps[4], dq, hq, sh.Nq, D, 128, bf16) && map16(&maps[5], dk, hk, sh.Nk, D, 128, bf16) &&
         map16(&maps[6], dv, hk, sh.Nk, D, 128, bf16) && map16(&maps[7], q, hq, sh.Nq, D, 128, bf16) &&
         map16(&maps[8], k, hk, sh.Nk, D, 64, bf16) && map16(&maps[9], o, hq, sh.Nq, D, 128, bf16);
}

void bwd_shape_params(fa::BwdParams& prm, const Shape& sh) {
  prm.heads = static_cast<int>(sh.q_heads());
  prm.group = sh.group();
  prm.Nq = sh.Nq;
  prm.Nk = sh.Nk;
  prm.Nq_pad = sh.nq_pad();
  prm.causal_off = sh.Nk - sh.Nq;
}

// The backward launch sequence, once the arguments passed their checks:
// `scratch` holds the [delta | lse2] layout of `ws` (a caller workspace or the
// library's built-in buffer).  Every entry point maps launch failures the
// same way: FA_OK or FA_ERR_CUDA.
int bwd_run(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, char* scratch, const BwdWorkspace& ws, const Shape& sh, float scale,
            cudaStream_t stream, bool bf16, const DevInfo* dev) {
  CUtensorMap maps[kBwdMaps];
  if (!bwd_maps(maps, q, k, v, o, dout, dq, dk, dv, sh, bf16)) return FA_ERR_CUDA;
  fa::BwdParams prm{};
  prm.v = static_cast<const __half*>(v);
  prm.o = static_cast<const __half*>(o);
  prm.dout = static_cast<const __half*>(dout);
  prm.lse = lse;
  prm.dq = static_cast<__half*>(dq);
  prm.dk = static_cast<__half*>(dk);
  prm.dv = static_cast<__half*>(dv);
  prm.delta = reinterpret_cast<float*>(scratch + ws.delta_off);
  prm.lse2 = reinterpret_cast<float*>(scratch + ws.lse2_off);
  bwd_shape_params(prm, sh);
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  prm.status = dev->status;
  const bool c = sh.causal != 0;
  int rc;
  switch (sh.D) {
    case 64: rc = fa::launch_bwd_d64(c, bf16, maps, prm, dev->sms, stream); break;
    case 128: rc = fa::launch_bwd_d128(c, bf16, maps, prm, dev->sms, stream); break;
    default: rc = fa::launch_bwd_d256(c, bf16, maps, prm, dev->sms, stream); break;
  }
  return rc == 0 ? FA_OK : FA_ERR_CUDA;
}

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, const Shape& sh, float scale,
             cudaStream_t stream, bool bf16) {
  int rc = bwd_checks(q, k, v, o, dout, lse, dq, dk, dv, sh, scale);
  if (rc != FA_OK) return rc;
  DevInfo* dev = nullptr;
  if ((rc = current_device_info(&dev)) != FA_OK) return rc;
  const BwdWorkspace ws = bwd_workspace_layout(sh);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < ws.total) return FA_ERR_WORKSPACE;
  return bwd_run(q, k, v, o, dout, lse, dq, dk, dv, static_cast<char*>(workspace), ws, sh, scale, stream, bf16, dev);
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int Z, int H, int N, int D,
           int causal, float scale, cudaStream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, square(Z, H, N, D, causal), scale,
                  stream, false);
}

int fa_bwd_bf16(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int Z, int H, int N, int D,
                int causal, float scale, cudaStream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, square(Z, H, N, D, causal), scale,
                  stream, true);
}

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
              void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int Z, int H, int Hkv, int Nq,
              int Nk, int D, int causal, float scale, int dtype, cudaStream_t stream) {
  if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, Shape{Z, H, Hkv, Nq, Nk, D, causal},
                  scale, stream, dtype == FA_DTYPE_BF16);
}

int fa_device_status_raw(cudaStream_t stream, int* raw) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  DevInfo* dev = nullptr;
  int rc = current_device_info(&dev);
  if (rc != FA_OK) return rc;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (raw) *raw = v;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

int fa_device_status(cudaStream_t stream) { return fa_device_status_raw(stream, nullptr); }

}  // extern "C"

// ---------------------------------------------------------------------------
// fa_bwd_noalloc: the backward for callers that cannot allocate device
// memory.  Its scratch is this file-scope buffer instead of a caller
// workspace.  In host code `g_fa_noalloc_scratch` names a host-side shadow,
// not the device buffer, so the device address is looked up once per device
// with cudaGetSymbolAddress and only that address is handed to the kernels.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the built-in buffer on the current device (first call on
// a device looks it up).  Returns nullptr on failure.
void* noalloc_scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}
}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int Z, int H, int N, int D,
                              int causal, float scale, cudaStream_t stream) {
  const Shape sh = square(Z, H, N, D, causal);
  int rc = bwd_checks(q, k, v, o, dout, lse, dq, dk, dv, sh, scale);
  if (rc != FA_OK) return rc;
  DevInfo* dev = nullptr;
  if ((rc = current_device_info(&dev)) != FA_OK) return rc;

  // Scratch layout [delta | lse2], as fa_bwd's workspace.
  const BwdWorkspace ws = bwd_workspace_layout(sh);
  if (ws.total > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;

  char* scratch = static_cast<char*>(noalloc_scratch_on_current_device());
  if (scratch == nullptr) return FA_ERR_CUDA;

  return bwd_run(q, k, v, o, dout, lse, dq, dk, dv, scratch, ws, sh, scale, stream, false, dev);
}

extern "C" int fa_selftest_wait_timeout(cudaStream_t stream) {
  DevInfo* dev = nullptr;
  int rc = current_device_info(&dev);
  if (rc != FA_OK) return rc;
  fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(dev->status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
