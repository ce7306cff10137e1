// Exported C ABI (include/moe_mxfp4.h): argument checks on the host, workspace
// carving, and the launch sequence of each entry point on the caller's stream.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include <cuda_runtime.h>

#include "../../include/moe_mxfp4.h"
#include "decode_mx.cuh"
#include "moe_internal.h"

namespace moe {

// Per device: [0] MOE_STATUS_* bits, [1] the first timeout site (moe_get_timeout_site).
__device__ int g_status_word[2];

static std::atomic<uint64_t> g_launches{0};
static thread_local int t_last_cuda_error = 0;

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void set_last_cuda_error(int err) { t_last_cuda_error = err; }

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sms = 0;
  int* status = nullptr;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// Probes the current device once: architecture, SM count, status-word address.
int current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    t_last_cuda_error = (int)err;
    return MOE_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
      t_last_cuda_error = (int)err;
      return MOE_ECUDA;
    }
    void* p = nullptr;
    if ((err = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) {
      t_last_cuda_error = (int)err;
      return MOE_ECUDA;
    }
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    d.status = static_cast<int*>(p);
    d.probed = true;
  }
  if (!d.supported) return MOE_EUNSUPPORTED;
  *out = &d;
  return MOE_OK;
}

int cuda_status(cudaError_t err) {
  if (err == cudaSuccess) return MOE_OK;
  t_last_cuda_error = (int)err;
  return MOE_ECUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t max_rows_of(int T, int k, int E, int tile) {
  const size_t n = (size_t)T * k + (size_t)E * (tile - 1);
  return round_up(n, (size_t)tile);
}

int resolve_rail(int T, int rail) {
  if (rail == MOE_RAIL_AUTO)
    return T <= MOE_AUTO_GEMV_MAX_T ? MOE_RAIL_GEMV : T <= MOE_AUTO_MX_MAX_T ? MOE_RAIL_GROUPED_MX : MOE_RAIL_GROUPED_MM;
  return rail;
}

struct Workspace {
  float* logits;
  float* rpart;    // grouped rails: the split router's partial dots
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* basep;
  int32_t* rows;
  int32_t* inv;
  float* h;        // GEMV rail: [T*k][F] pair-swizzled
  uint16_t* xg;    // grouped rail: [max_rows][D] bf16, high parts of x
  uint16_t* xg_lo; // grouped rail: [max_rows][D] bf16, low parts of x
  uint16_t* hg;    // grouped rail: [max_rows][F] bf16
  // block-scaled rail: E4M3 operand terms in bucket order and their scale words
  uint8_t* xq;       // [kMxXTerms][max_rows][D]
  uint32_t* xs;      // [kMxXTerms][D/128 rounded up][max_rows]
  uint8_t* hq;       // [kMxHTerms][max_rows][F]
  uint32_t* hs;      // [kMxHTerms][F/128 rounded up][max_rows]
  // Q8 rail
  int8_t* x8;        // [T][D]
  float* xd;         // [T][D/32]
  float* gq;         // [T*k][F] gate, then h
  float* uq;         // [T*k][F]
  int8_t* h8;        // [T*k][F]
  float* hd;         // [T*k][F/32]
  float* od;         // [T*k][D] down rows + bias, per slot
  size_t max_rows;
};

// Lays the workspace out from `base` (nullptr: size only). Returns total bytes.
size_t layout_workspace(int T, int D, int F, int E, int k, int rail, char* base, Workspace* ws) {
  const int tile = (rail == MOE_RAIL_GEMV || rail == MOE_RAIL_GEMV_Q8) ? 1 : MOE_MM_TILE;
  const size_t mr = max_rows_of(T, k, E, tile);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = round_up(off + bytes, 256);
    return p;
  };
  Workspace w{};
  w.logits = reinterpret_cast<float*>(take((size_t)T * E * 4));
  if (tile != 1) w.rpart = reinterpret_cast<float*>(take(router_partials_bytes(T, E)));
  w.ids = reinterpret_cast<int32_t*>(take((size_t)T * k * 4));
  w.w = reinterpret_cast<float*>(take((size_t)T * k * 4));
  w.counts = reinterpret_cast<int32_t*>(take((size_t)E * 4));
  w.basep = reinterpret_cast<int32_t*>(take((size_t)(E + 1) * 4));
  w.rows = reinterpret_cast<int32_t*>(take(mr * 4));
  w.inv = reinterpret_cast<int32_t*>(take((size_t)T * k * 4));
  if (rail == MOE_RAIL_GEMV) {
    w.h = reinterpret_cast<float*>(take((size_t)T * k * F * 4));
  } else if (rail == MOE_RAIL_GEMV_Q8) {
    const size_t TK = (size_t)T * k;
    w.x8 = reinterpret_cast<int8_t*>(take((size_t)T * D));
    w.xd = reinterpret_cast<float*>(take((size_t)T * (D / 32) * 4));
    w.gq = reinterpret_cast<float*>(take(TK * F * 4));
    w.uq = reinterpret_cast<float*>(take(TK * F * 4));
    w.h8 = reinterpret_cast<int8_t*>(take(TK * F));
    w.hd = reinterpret_cast<float*>(take(TK * (F / 32) * 4));
    w.od = reinterpret_cast<float*>(take(TK * D * 4));
  } else if (rail == MOE_RAIL_GROUPED_MX) {
    const size_t nd = (size_t)(D / 32 + 3) / 4, nf = (size_t)(F / 32 + 3) / 4;
    w.xq = reinterpret_cast<uint8_t*>(take(kMxXTerms * mr * D));
    w.xs = reinterpret_cast<uint32_t*>(take(kMxXTerms * nd * mr * 4));
    w.hq = reinterpret_cast<uint8_t*>(take(kMxHTerms * mr * F));
    w.hs = reinterpret_cast<uint32_t*>(take(kMxHTerms * nf * mr * 4));
  } else {
    w.xg = reinterpret_cast<uint16_t*>(take(mr * D * 2));
    w.xg_lo = reinterpret_cast<uint16_t*>(take(mr * D * 2));
    w.hg = reinterpret_cast<uint16_t*>(take(mr * F * 2));
  }
  w.max_rows = mr;
  if (ws) *ws = w;
  return off;
}

// Workspace of the block-scaled decode rail on prepacked weights.
struct PackedWorkspace {
  float* logits;  // [T][E]
  uint8_t* xq;    // x operand chunks [NK_D][npad][64]
  uint8_t* xsf;   // [NK_D][512]
  uint8_t* hq;    // down operand chunks [T*k][NK_F][npad][64]
  uint8_t* hsf;   // [T*k][NK_F][512]
  float* part;    // partial sums [kDecodeMxMaxGrid][2][2][T][128]
  int* cnt;       // arrival counters per unit and lane quarter: gate/up [T*k*NK_F][4], then down [NK_D][4]
  int ncnt_gu, ncnt;
  float* xs;      // host-I/O staging [T][D]
  float* ys;      // [T][D]
};

size_t layout_packed_workspace(int T, int D, int F, int k, int E, char* base, PackedWorkspace* ws) {
  const int npad = dmx::npad_for(T);
  const size_t nkd = (size_t)(D + 127) / 128, nkf = (size_t)(F + 127) / 128;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = round_up(off + bytes, 256);
    return p;
  };
  PackedWorkspace w{};
  w.logits = reinterpret_cast<float*>(take((size_t)T * E * 4));
  w.xq = reinterpret_cast<uint8_t*>(take(nkd * npad * 64));
  w.xsf = reinterpret_cast<uint8_t*>(take(nkd * 512));
  w.hq = reinterpret_cast<uint8_t*>(take((size_t)T * k * nkf * npad * 64));
  w.hsf = reinterpret_cast<uint8_t*>(take((size_t)T * k * nkf * 512));
  w.part = reinterpret_cast<float*>(take((size_t)kDecodeMxMaxGrid * 2 * 2 * T * 128 * 4));
  w.ncnt_gu = (int)(4 * (size_t)T * k * nkf);  // one counter per unit and lane quarter
  w.ncnt = w.ncnt_gu + 4 * (int)nkd;
  w.cnt = reinterpret_cast<int*>(take((size_t)w.ncnt * 4));
  w.xs = reinterpret_cast<float*>(take((size_t)T * D * 4));
  w.ys = reinterpret_cast<float*>(take((size_t)T * D * 4));
  if (ws) *ws = w;
  return off;
}

int resolve_packed_rail(int T, int rail) {
  if (rail == MOE_RAIL_AUTO) return T <= MOE_AUTO_DECODE_MX_MAX_T ? MOE_RAIL_DECODE_MX : MOE_RAIL_GROUPED_MX4;
  return rail;
}

// Workspace of the prefill rail on prepacked weights (MOE_RAIL_GROUPED_MX4).
struct PackedPrefillWorkspace {
  float* logits;
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* basep;
  int32_t* rows;
  int32_t* inv;
  uint8_t* aq;   // x terms in bucket order, activation-chunk layout
  uint8_t* asf;
  float* rpart;  // the split router's partial dots
  int2* segs;    // segment table of the bucket
  int* ctr;      // the two GEMMs' unit counters
  float* hf;     // h as float rows, written by the gate/up GEMM
  uint8_t* hq;   // h terms
  uint8_t* hsf;
  float* xs;     // host-I/O staging [T][D]
  float* ys;
  size_t max_rows;
};

size_t layout_packed_prefill_workspace(int T, int D, int F, int k, int E, char* base, PackedPrefillWorkspace* ws) {
  const size_t mr = max_rows_of(T, k, E, MOE_MM_TILE);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = round_up(off + bytes, 256);
    return p;
  };
  PackedPrefillWorkspace w{};
  w.logits = reinterpret_cast<float*>(take((size_t)T * E * 4));
  w.ids = reinterpret_cast<int32_t*>(take((size_t)T * k * 4));
  w.w = reinterpret_cast<float*>(take((size_t)T * k * 4));
  w.counts = reinterpret_cast<int32_t*>(take((size_t)E * 4));
  w.basep = reinterpret_cast<int32_t*>(take((size_t)(E + 1) * 4));
  w.rows = reinterpret_cast<int32_t*>(take(mr * 4));
  w.inv = reinterpret_cast<int32_t*>(take((size_t)T * k * 4));
  w.aq = reinterpret_cast<uint8_t*>(take(prefill_operand_bytes((int)mr, D, kPrefillXTerms)));
  w.asf = reinterpret_cast<uint8_t*>(take(prefill_atom_bytes((int)mr, D, kPrefillXTerms)));
  w.rpart = reinterpret_cast<float*>(take(router_partials_bytes(T, E)));
  w.segs = reinterpret_cast<int2*>(take((2 * (mr / 128) + 1) * sizeof(int2)));
  w.ctr = reinterpret_cast<int*>(take(2 * sizeof(int)));
  w.hf = reinterpret_cast<float*>(take(mr * (size_t)F * 4));
  w.hq = reinterpret_cast<uint8_t*>(take(prefill_operand_bytes((int)mr, F, kPrefillHTerms)));
  w.hsf = reinterpret_cast<uint8_t*>(take(prefill_atom_bytes((int)mr, F, kPrefillHTerms)));
  w.xs = reinterpret_cast<float*>(take((size_t)T * D * 4));
  w.ys = reinterpret_cast<float*>(take((size_t)T * D * 4));
  w.max_rows = mr;
  if (ws) *ws = w;
  return off;
}

}  // namespace

int device_sm_count() {
  DeviceInfo* d = nullptr;
  if (current_device(&d) != MOE_OK) return 1;
  return d->sms;
}

namespace {
std::mutex g_fn_mu;
std::map<std::pair<const void*, int>, size_t> g_smem_set;
std::map<std::tuple<const void*, int, int, size_t>, int> g_resident;
}  // namespace

cudaError_t ensure_smem_limit_fn(const void* kern, size_t bytes) {
  if (bytes == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_fn_mu);
  auto key = std::make_pair(kern, dev);
  auto it = g_smem_set.find(key);
  if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (err == cudaSuccess) g_smem_set[key] = bytes;
  return err;
}

int resident_blocks_per_sm_fn(const void* kern, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  std::lock_guard<std::mutex> lock(g_fn_mu);
  auto key = std::make_tuple(kern, dev, threads, smem);
  auto it = g_resident.find(key);
  if (it != g_resident.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess || n < 1) n = 1;
  g_resident[key] = n;
  return n;
}

}  // namespace moe

using namespace moe;

#define MOE_REQUIRE(cond)              \
  do {                                 \
    if (!(cond)) return MOE_EINVAL;    \
  } while (0)

extern "C" {

size_t moe_bucket_max_rows(int T, int k, int E, int tile) {
  if (T < 0 || k < 1 || E < 1 || tile < 1) return 0;
  return max_rows_of(T, k, E, tile);
}

size_t moe_ffn_workspace_bytes(int T, int D, int F, int E, int k, int rail) {
  if (T < 0 || D < 1 || F < 1 || E < 1 || k < 1 || k > E) return 0;
  rail = resolve_rail(T, rail);
  if (rail != MOE_RAIL_GEMV && rail != MOE_RAIL_GROUPED_MM && rail != MOE_RAIL_GROUPED_MX &&
      rail != MOE_RAIL_GEMV_Q8)
    return 0;
  if (rail == MOE_RAIL_GEMV_Q8 && (T > MOE_GEMV_MAX_T || D % 32 || F % 32)) return 0;
  return layout_workspace(T, D, F, E, k, rail, nullptr, nullptr);
}

int moe_route_topk(const float* x, int T, int D, const float* w_router, const float* b_router,
                   int E, int k, float* logits, int32_t* ids, float* weights, cudaStream_t stream) {
  MOE_REQUIRE(T >= 0 && D >= 4 && D % 4 == 0);
  MOE_REQUIRE(E >= 1 && E <= 256 && k >= 1 && k <= E && k <= 32);
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && w_router && logits && ids && weights);
  MOE_REQUIRE(aligned(x, 16) && aligned(w_router, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  rc = cuda_status(launch_router_logits(x, T, D, w_router, b_router, E, logits, nullptr, L));
  if (rc != MOE_OK) return rc;
  L.pdl = true;
  return cuda_status(launch_topk_softmax(logits, T, E, k, ids, weights, L));
}

int moe_bucket(const int32_t* ids, int T, int k, int E, int tile, int32_t* counts, int32_t* basep,
               int32_t* rows, int32_t* inv, cudaStream_t stream) {
  MOE_REQUIRE(T >= 0 && k >= 1 && E >= 1 && E <= 1024 && tile >= 1 && tile <= 1024);
  MOE_REQUIRE(counts && basep && rows && (T == 0 || (ids && inv)));
  MOE_REQUIRE((size_t)T * k + (size_t)E * tile < (size_t)1 << 30);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  const int mr = (int)max_rows_of(T, k, E, tile);
  return cuda_status(launch_bucket(ids, T, k, E, tile, mr, counts, basep, rows, inv, d->status, L));
}

int moe_mxfp4_gemv(const uint8_t* w_qs, const uint8_t* w_sc, int E, int R, int C,
                   const int32_t* experts, int n, const float* x, int64_t x_stride,
                   const float* bias, float* out, cudaStream_t stream) {
  MOE_REQUIRE(E >= 1 && R >= 1 && C >= 32 && C % 32 == 0 && n >= 0 && x_stride >= 0);
  MOE_REQUIRE(x_stride % 4 == 0);
  if (n == 0) return MOE_OK;
  if (C > 4096) return MOE_EUNSUPPORTED;
  MOE_REQUIRE(w_qs && w_sc && experts && x && out);
  MOE_REQUIRE(aligned(w_qs, 16) && aligned(x, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(
      launch_mxfp4_gemv(w_qs, w_sc, E, R, C, experts, n, x, x_stride, bias, out, d->status, L));
}

int moe_quantize_q8(const float* x, int64_t rows, int C, int8_t* q, float* d, cudaStream_t stream) {
  MOE_REQUIRE(rows >= 0 && C >= 32 && C % 32 == 0);
  if (rows == 0) return MOE_OK;
  MOE_REQUIRE(x && q && d && aligned(x, 16) && aligned(q, 16));
  DeviceInfo* dv = nullptr;
  int rc = current_device(&dv);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_quant_q8(x, rows, C, q, d, L));
}

int moe_mxfp4_gemv_q8(const uint8_t* w_qs, const uint8_t* w_sc, int E, int R, int C, const int32_t* experts,
                      int n, int act_div, const int8_t* q, const float* d, const float* bias, float* out,
                      cudaStream_t stream) {
  MOE_REQUIRE(E >= 1 && R >= 1 && C >= 32 && C % 32 == 0 && n >= 0 && act_div >= 1);
  if (n == 0) return MOE_OK;
  if (C > 4096) return MOE_EUNSUPPORTED;
  MOE_REQUIRE(w_qs && w_sc && experts && q && d && out);
  MOE_REQUIRE(aligned(w_qs, 16) && aligned(q, 16));
  DeviceInfo* dv = nullptr;
  int rc = current_device(&dv);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_gemv_q8(w_qs, w_sc, E, R, C, experts, n, act_div, q, d, bias, out, dv->status, L));
}

int moe_swiglu_oai(const float* g, const float* u, void* h, int64_t n, int h_dtype, float alpha,
                   float limit, cudaStream_t stream) {
  MOE_REQUIRE(n >= 0 && (h_dtype == MOE_DTYPE_F32 || h_dtype == MOE_DTYPE_BF16));
  if (n == 0) return MOE_OK;
  MOE_REQUIRE(g && u && h);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_swiglu(g, u, h, n, h_dtype, alpha, limit, L));
}

int moe_selftest_wait_timeout(const void* src, cudaStream_t stream) {
  MOE_REQUIRE(src && aligned(src, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_selftest_wait_timeout(static_cast<const uint8_t*>(src), d->status, L));
}

int moe_rms_renorm(const float* x, int T, int D, float* y, cudaStream_t stream) {
  MOE_REQUIRE(T >= 0 && D >= 1);
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && y);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_rms_renorm(x, T, D, y, L));
}

int moe_gather_rows_bf16(const float* x, int T, int D, int k, const int32_t* rows,
                         const int32_t* basep, int E, int max_rows, uint16_t* xg, uint16_t* xg_lo,
                         float* y_zero, cudaStream_t stream) {
  MOE_REQUIRE(T >= 0 && D >= 8 && D % 8 == 0 && k >= 1 && E >= 1 && max_rows >= 0);
  MOE_REQUIRE(rows && basep && xg && (T == 0 || x));
  MOE_REQUIRE(aligned(x, 16) && aligned(xg, 16) && aligned(xg_lo, 16) && aligned(y_zero, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_gather_bf16(x, T, D, k, rows, basep, E, max_rows, xg, xg_lo, y_zero, true, L));
}

int moe_mxfp4_grouped_mm(const uint8_t* w_qs, const uint8_t* w_sc, const float* bias,
                         const uint8_t* w2_qs, const uint8_t* w2_sc, const float* bias2, int E,
                         int R, int C, const uint16_t* a, const uint16_t* a_lo,
                         const int32_t* counts, const int32_t* basep, const int32_t* rows,
                         int max_rows, int k, const float* weights, int epilogue, float alpha,
                         float limit, void* out, int64_t out_ld, cudaStream_t stream) {
  MOE_REQUIRE(E >= 1 && E <= 1024 && R >= 1 && C >= 64 && k >= 1 && max_rows >= 0);
  MOE_REQUIRE(epilogue == MOE_EPI_STORE_BF16 || epilogue == MOE_EPI_SWIGLU_BF16 ||
              epilogue == MOE_EPI_SCATTER_WEIGHTED);
  MOE_REQUIRE(max_rows % MOE_MM_TILE == 0);
  if (C % 64 != 0 || C > 4096 || R % 8 != 0) return MOE_EUNSUPPORTED;
  MOE_REQUIRE(out_ld >= R && out_ld % 8 == 0);
  MOE_REQUIRE(w_qs && w_sc && a && counts && basep && rows && out);
  MOE_REQUIRE(aligned(w_qs, 16) && aligned(w_sc, 16) && aligned(a, 16) && aligned(a_lo, 16));
  if (epilogue == MOE_EPI_SWIGLU_BF16) {
    MOE_REQUIRE(w2_qs && w2_sc && aligned(w2_qs, 16) && aligned(w2_sc, 16));
  }
  if (epilogue == MOE_EPI_SCATTER_WEIGHTED) MOE_REQUIRE(weights != nullptr);
  if (max_rows == 0) return MOE_OK;
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  GroupedMMArgs g{};
  g.w_qs[0] = w_qs;
  g.w_sc[0] = w_sc;
  g.bias[0] = bias;
  g.w_qs[1] = w2_qs;
  g.w_sc[1] = w2_sc;
  g.bias[1] = bias2;
  g.nmat = (epilogue == MOE_EPI_SWIGLU_BF16) ? 2 : 1;
  g.E = E;
  g.R = R;
  g.C = C;
  g.a = a;
  g.a_lo = a_lo;
  g.counts = counts;
  g.basep = basep;
  g.rows = rows;
  g.max_rows = max_rows;
  g.k = k;
  g.weights = weights;
  g.epilogue = epilogue;
  g.alpha = alpha;
  g.limit = limit;
  g.out = out;
  g.out_ld = out_ld;
  g.out_rows = epilogue == MOE_EPI_SCATTER_WEIGHTED ? 0 : max_rows;  // the scatter's token count is not passed
  g.status = d->status;
  Launch L{stream, false};
  return cuda_status(launch_grouped_mm(g, L));
}

int moe_expert_gateup_swiglu(const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                             const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, int E,
                             int F, int D, int T, int k, const float* x, const int32_t* ids,
                             float alpha, float limit, float* h, cudaStream_t stream) {
  MOE_REQUIRE(T >= 0 && T <= MOE_GEMV_MAX_T && k >= 1 && k <= 8 && E >= 1 && E <= 256);
  MOE_REQUIRE(D >= 64 && F >= 64 && D % 64 == 0 && F % 64 == 0);
  if (D > 4096 || F > 4096) return MOE_EUNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(g_qs && g_sc && u_qs && u_sc && x && ids && h);
  MOE_REQUIRE(aligned(g_qs, 16) && aligned(u_qs, 16) && aligned(x, 16) && aligned(h, 16));
  MOE_REQUIRE(aligned(g_sc, 16) && aligned(u_sc, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_gemv_gateup(g_qs, g_sc, bg, u_qs, u_sc, bu, E, F, D, T, k, x, nullptr,
                                        ids, nullptr, nullptr, alpha, limit, h, d->status, false, L));
}

int moe_expert_down_combine(const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int E, int D,
                            int F, int T, int k, const float* h, const int32_t* ids,
                            const float* weights, float* y, cudaStream_t stream) {
  MOE_REQUIRE(T >= 0 && T <= MOE_GEMV_MAX_T && k >= 1 && k <= 8 && E >= 1 && E <= 256);
  MOE_REQUIRE(D >= 64 && F >= 64 && D % 64 == 0 && F % 64 == 0);
  if (D > 4096 || F > 4096) return MOE_EUNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(d_qs && d_sc && h && ids && weights && y);
  MOE_REQUIRE(aligned(d_qs, 16) && aligned(d_sc, 16) && aligned(h, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_gemv_down(d_qs, d_sc, bd, E, D, F, T, k, h, nullptr, ids, weights, y,
                                      d->status, L));
}

}  // extern "C"

namespace {
// moe_ffn_layer with an optional device copy of x made by the router on the
// GEMV rail (x may then live in mapped host memory: it is read once).
int ffn_layer_impl(const float* x, float* x_copy, int T, int D, int F, int E, int k, const float* w_router,
                  const float* b_router, const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                  const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, const uint8_t* d_qs,
                  const uint8_t* d_sc, const float* bd, int rail, void* workspace,
                  size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out,
                  cudaStream_t stream, int gu_rs = 1) {
  // gu_rs = 2: gate and up are one plane with interleaved rows; u_qs, u_sc, bu
  // point one row (or one bias) past g_qs, g_sc, bg
  MOE_REQUIRE(T >= 0 && D >= 64 && F >= 64 && D % 64 == 0 && F % 64 == 0);
  MOE_REQUIRE(E >= 1 && E <= 256 && k >= 1 && k <= E && k <= 32);
  rail = resolve_rail(T, rail);
  MOE_REQUIRE(rail == MOE_RAIL_GEMV || rail == MOE_RAIL_GROUPED_MM || rail == MOE_RAIL_GROUPED_MX ||
              rail == MOE_RAIL_GEMV_Q8);
  if (rail == MOE_RAIL_GEMV || rail == MOE_RAIL_GEMV_Q8) {
    MOE_REQUIRE(T <= MOE_GEMV_MAX_T && k <= 8);
    if (D > 4096 || F > 4096) return MOE_EUNSUPPORTED;
  } else {
    if (D > 4096 || F > 4096) return MOE_EUNSUPPORTED;
  }
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && w_router && g_qs && g_sc && u_qs && u_sc && d_qs && d_sc && y && workspace);
  MOE_REQUIRE(aligned(x, 16) && aligned(w_router, 16) && aligned(y, 16) && aligned(workspace, 256));
  MOE_REQUIRE(aligned(g_qs, 16) && aligned(u_qs, 16) && aligned(d_qs, 16));
  MOE_REQUIRE(aligned(g_sc, 16) && (gu_rs == 2 || aligned(u_sc, 16)) && aligned(d_sc, 16));
  const size_t need = layout_workspace(T, D, F, E, k, rail, nullptr, nullptr);
  MOE_REQUIRE(workspace_bytes >= need);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Workspace ws;
  layout_workspace(T, D, F, E, k, rail, static_cast<char*>(workspace), &ws);
  int32_t* ids = ids_out ? ids_out : ws.ids;
  float* wts = weights_out ? weights_out : ws.w;
  const float alpha = 1.702f, limit = 7.0f;

  Launch L{stream, false};
  if (rail != MOE_RAIL_GEMV) x_copy = nullptr;  // prefill sizes read x from device memory
  MOE_REQUIRE(x_copy == nullptr || aligned(x_copy, 16));
  if (ws.rpart) {  // grouped rails: router split over D, then top-k
    if ((rc = cuda_status(launch_route_topk(x, T, D, w_router, b_router, E, k, ws.logits, ws.rpart, ids, wts, L))) !=
        MOE_OK)
      return rc;
    L.pdl = true;
  } else {
    rc = cuda_status(launch_router_logits(x, T, D, w_router, b_router, E, ws.logits, x_copy, L));
    if (rc != MOE_OK) return rc;
    L.pdl = true;
  }
  if (rail == MOE_RAIL_GEMV) {
    // decode: the two expert kernels take the top-k of the logits themselves
    rc = cuda_status(launch_gemv_gateup(g_qs, g_sc, bg, u_qs, u_sc, bu, E, F, D, T, k, x_copy ? x_copy : x,
                                        ws.logits, nullptr, ids_out, weights_out, alpha, limit, ws.h, d->status,
                                        x_copy != nullptr, L, gu_rs));
    if (rc != MOE_OK) return rc;
    return cuda_status(launch_gemv_down(d_qs, d_sc, bd, E, D, F, T, k, ws.h, ws.logits, nullptr,
                                        nullptr, y, d->status, L));
  }
  if (!ws.rpart && (rc = cuda_status(launch_topk_softmax(ws.logits, T, E, k, ids, wts, L))) != MOE_OK) return rc;
  if (rail == MOE_RAIL_GEMV_Q8) {
    // x -> Q8; gate and up per slot (the slot's token row); swiglu in place; h -> Q8; down per slot; combine
    const int TK = T * k;
    if ((rc = cuda_status(launch_quant_q8(x, T, D, ws.x8, ws.xd, L))) != MOE_OK) return rc;
    if ((rc = cuda_status(launch_gemv_q8(g_qs, g_sc, E, F, D, ids, TK, k, ws.x8, ws.xd, bg, ws.gq, d->status, L, gu_rs))) !=
        MOE_OK)
      return rc;
    if ((rc = cuda_status(launch_gemv_q8(u_qs, u_sc, E, F, D, ids, TK, k, ws.x8, ws.xd, bu, ws.uq, d->status, L, gu_rs))) !=
        MOE_OK)
      return rc;
    if ((rc = cuda_status(launch_swiglu(ws.gq, ws.uq, ws.gq, (int64_t)TK * F, MOE_DTYPE_F32, alpha, limit, L))) !=
        MOE_OK)
      return rc;
    if ((rc = cuda_status(launch_quant_q8(ws.gq, TK, F, ws.h8, ws.hd, L))) != MOE_OK) return rc;
    if ((rc = cuda_status(launch_gemv_q8(d_qs, d_sc, E, D, F, ids, TK, 1, ws.h8, ws.hd, bd, ws.od, d->status, L))) !=
        MOE_OK)
      return rc;
    return cuda_status(launch_combine_slots(ws.od, wts, ids, T, k, D, E, y, L));
  }
  rc = cuda_status(launch_bucket(ids, T, k, E, MOE_MM_TILE, (int)ws.max_rows, ws.counts, ws.basep,
                                 ws.rows, ws.inv, d->status, L));
  if (rc != MOE_OK) return rc;
  if (rail == MOE_RAIL_GROUPED_MX) {
    rc = cuda_status(launch_quant_rows_mx(x, T, D, k, ws.rows, ws.basep, E, (int)ws.max_rows, ws.xq, ws.xs, y,
                                          L));
    if (rc != MOE_OK) return rc;
    GroupedMXArgs g{};
    g.w_qs[0] = g_qs;
    g.w_sc[0] = g_sc;
    g.bias[0] = bg;
    g.w_qs[1] = u_qs;
    g.w_sc[1] = u_sc;
    g.bias[1] = bu;
    g.nmat = 2;
    g.E = E;
    g.R = F;
    g.C = D;
    g.a_terms = ws.xq;
    g.a_sc = ws.xs;
    g.counts = ws.counts;
    g.basep = ws.basep;
    g.rows = ws.rows;
    g.max_rows = (int)ws.max_rows;
    g.k = k;
    g.weights = wts;
    g.alpha = alpha;
    g.limit = limit;
    g.h_terms = ws.hq;
    g.h_sc = ws.hs;
    g.status = d->status;
    g.rs = gu_rs;
    rc = cuda_status(launch_grouped_mx(g, L));
    if (rc != MOE_OK) return rc;
    GroupedMXArgs gd = g;
    gd.rs = 1;
    gd.w_qs[0] = d_qs;
    gd.w_sc[0] = d_sc;
    gd.bias[0] = bd;
    gd.w_qs[1] = nullptr;
    gd.w_sc[1] = nullptr;
    gd.bias[1] = nullptr;
    gd.nmat = 1;
    gd.R = D;
    gd.C = F;
    gd.a_terms = ws.hq;
    gd.a_sc = ws.hs;
    gd.h_terms = nullptr;
    gd.h_sc = nullptr;
    gd.y = y;
    return cuda_status(launch_grouped_mx(gd, L));
  }
  rc = cuda_status(launch_gather_bf16(x, T, D, k, ws.rows, ws.basep, E, (int)ws.max_rows, ws.xg,
                                      ws.xg_lo, y, false, L));
  if (rc != MOE_OK) return rc;
  GroupedMMArgs g{};
  g.w_qs[0] = g_qs;
  g.w_sc[0] = g_sc;
  g.bias[0] = bg;
  g.w_qs[1] = u_qs;
  g.w_sc[1] = u_sc;
  g.bias[1] = bu;
  g.nmat = 2;
  g.E = E;
  g.R = F;
  g.C = D;
  g.a = ws.xg;
  g.a_lo = ws.xg_lo;  // gate/up on split activations: x = hi + lo (16 significant bits)
  g.counts = ws.counts;
  g.basep = ws.basep;
  g.rows = ws.rows;
  g.max_rows = (int)ws.max_rows;
  g.k = k;
  g.weights = wts;
  g.epilogue = MOE_EPI_SWIGLU_BF16;
  g.alpha = alpha;
  g.limit = limit;
  g.out = ws.hg;
  g.out_ld = F;
  g.out_rows = (int64_t)ws.max_rows;
  g.status = d->status;
  g.rs = gu_rs;
  rc = cuda_status(launch_grouped_mm(g, L));
  if (rc != MOE_OK) return rc;
  GroupedMMArgs gd = g;
  gd.rs = 1;
  gd.w_qs[0] = d_qs;
  gd.w_sc[0] = d_sc;
  gd.bias[0] = bd;
  gd.w_qs[1] = nullptr;
  gd.w_sc[1] = nullptr;
  gd.bias[1] = nullptr;
  gd.nmat = 1;
  gd.R = D;
  gd.C = F;
  gd.a = ws.hg;
  gd.a_lo = nullptr;  // h enters the down projection as plain bf16
  gd.epilogue = MOE_EPI_SCATTER_WEIGHTED;
  gd.out = y;
  gd.out_ld = D;
  gd.out_rows = T;
  return cuda_status(launch_grouped_mm(gd, L));
}

}  // namespace

extern "C" {

int moe_ffn_layer(const float* x, int T, int D, int F, int E, int k, const float* w_router,
                  const float* b_router, const uint8_t* g_qs, const uint8_t* g_sc, const float* bg,
                  const uint8_t* u_qs, const uint8_t* u_sc, const float* bu, const uint8_t* d_qs,
                  const uint8_t* d_sc, const float* bd, int rail, void* workspace,
                  size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out,
                  cudaStream_t stream) {
  return ffn_layer_impl(x, nullptr, T, D, F, E, k, w_router, b_router, g_qs, g_sc, bg, u_qs, u_sc, bu, d_qs, d_sc,
                        bd, rail, workspace, workspace_bytes, y, ids_out, weights_out, stream);
}

int moe_ffn_layer_gu(const float* x, int T, int D, int F, int E, int k, const float* w_router,
                     const float* b_router, const uint8_t* gu_qs, const uint8_t* gu_sc, const float* gu_b,
                     const uint8_t* d_qs, const uint8_t* d_sc, const float* bd, int rail, void* workspace,
                     size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out, cudaStream_t stream) {
  MOE_REQUIRE(D >= 64 && D % 64 == 0);
  MOE_REQUIRE(T == 0 || (gu_qs && gu_sc));
  const uint8_t* u_qs = gu_qs ? gu_qs + D / 2 : nullptr;
  const uint8_t* u_sc = gu_sc ? gu_sc + D / 32 : nullptr;
  return ffn_layer_impl(x, nullptr, T, D, F, E, k, w_router, b_router, gu_qs, gu_sc, gu_b, u_qs, u_sc,
                        gu_b ? gu_b + 1 : nullptr, d_qs, d_sc, bd, rail, workspace, workspace_bytes, y, ids_out,
                        weights_out, stream, 2);
}

}  // extern "C"

namespace {
// Device address of pinned (page-locked, mapped) host memory, or nullptr for
// pageable memory.
const void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}
}  // namespace

extern "C" {

int moe_ffn_layer_hostio(const moe_ffn_args_t* args, const float* x_host, float* y_host,
                         cudaStream_t stream) {
  MOE_REQUIRE(args != nullptr);
  const moe_ffn_args_t& a = *args;
  MOE_REQUIRE(a.T >= 0 && a.D >= 64);
  if (a.T == 0) return MOE_OK;
  MOE_REQUIRE(x_host && y_host && a.x_dev && a.y_dev);
  if (resolve_rail(a.T, a.rail) == MOE_RAIL_GEMV) {
    // Decode rail with pinned buffers: no copies. The router reads x once from
    // host memory (over the CPU-GPU link) and leaves a copy in x_dev for the
    // gate/up kernel; the down kernel stores each element of y once, straight
    // into host memory.
    const float* dx = static_cast<const float*>(mapped_host(x_host));
    float* dy = static_cast<float*>(const_cast<void*>(mapped_host(y_host)));
    if (dx && dy)
      return ffn_layer_impl(dx, a.x_dev, a.T, a.D, a.F, a.E, a.k, a.w_router, a.b_router, a.g_qs, a.g_sc, a.bg,
                            a.u_qs, a.u_sc, a.bu, a.d_qs, a.d_sc, a.bd, a.rail, a.workspace, a.workspace_bytes,
                            dy, nullptr, nullptr, stream);
  }
  const size_t bytes = (size_t)a.T * a.D * sizeof(float);
  cudaError_t err = cudaMemcpyAsync(a.x_dev, x_host, bytes, cudaMemcpyHostToDevice, stream);
  if (err != cudaSuccess) return cuda_status(err);
  const int rc = moe_ffn_layer(a.x_dev, a.T, a.D, a.F, a.E, a.k, a.w_router, a.b_router, a.g_qs, a.g_sc,
                               a.bg, a.u_qs, a.u_sc, a.bu, a.d_qs, a.d_sc, a.bd, a.rail, a.workspace,
                               a.workspace_bytes, a.y_dev, nullptr, nullptr, stream);
  if (rc != MOE_OK) return rc;
  return cuda_status(cudaMemcpyAsync(y_host, a.y_dev, bytes, cudaMemcpyDeviceToHost, stream));
}

size_t moe_mxfp4_packed_qs_bytes(int E, int R, int C) {
  if (E < 1 || R < 1 || C < 32 || R % 64 != 0 || C % 32 != 0) return 0;
  return packed_qs_bytes(E, R, C);
}

size_t moe_mxfp4_packed_sf_bytes(int E, int R, int C) {
  if (E < 1 || R < 1 || C < 32 || R % 64 != 0 || C % 32 != 0) return 0;
  return packed_sf_bytes(E, R, C);
}

int moe_mxfp4_prepack(const uint8_t* qs, const uint8_t* sc, int E, int R, int C, uint8_t* qs_p,
                      uint8_t* sf_p, cudaStream_t stream) {
  MOE_REQUIRE(E >= 1 && R >= 64 && C >= 32 && R % 64 == 0 && C % 32 == 0);
  MOE_REQUIRE(qs && sc && qs_p && sf_p);
  MOE_REQUIRE(aligned(qs, 16) && aligned(sc, 16) && aligned(qs_p, 32) && aligned(sf_p, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  return cuda_status(launch_prepack(qs, sc, E, R, C, qs_p, sf_p, L));
}

int moe_mxfp4_prepack_gu(const uint8_t* gu_qs, const uint8_t* gu_sc, int E, int F, int D, uint8_t* g_qs_p,
                         uint8_t* g_sf_p, uint8_t* u_qs_p, uint8_t* u_sf_p, cudaStream_t stream) {
  MOE_REQUIRE(E >= 1 && F >= 64 && D >= 32 && F % 64 == 0 && D % 32 == 0);
  MOE_REQUIRE(gu_qs && gu_sc && g_qs_p && g_sf_p && u_qs_p && u_sf_p);
  MOE_REQUIRE(aligned(gu_qs, 16) && aligned(g_qs_p, 32) && aligned(u_qs_p, 32));
  MOE_REQUIRE(aligned(g_sf_p, 16) && aligned(u_sf_p, 16));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  Launch L{stream, false};
  rc = cuda_status(launch_prepack(gu_qs, gu_sc, E, F, D, g_qs_p, g_sf_p, L, 2));
  if (rc != MOE_OK) return rc;
  return cuda_status(launch_prepack(gu_qs + D / 2, gu_sc + D / 32, E, F, D, u_qs_p, u_sf_p, L, 2));
}

size_t moe_ffn_packed_workspace_bytes(int T, int D, int F, int E, int k, int rail) {
  if (T < 0 || D < 64 || F < 64 || D % 64 != 0 || F % 64 != 0 || E < 1 || k < 1 || k > E) return 0;
  rail = resolve_packed_rail(T, rail);
  if (rail == MOE_RAIL_GROUPED_MX4) return layout_packed_prefill_workspace(T, D, F, k, E, nullptr, nullptr);
  if (rail != MOE_RAIL_DECODE_MX || T > MOE_GEMV_MAX_T) return 0;
  return layout_packed_workspace(T, D, F, k, E, nullptr, nullptr);
}

}  // extern "C"

namespace {
// The prefill chain on prepacked planes: router, top-k, bucket (128-row tiles),
// x as E2M1 terms in bucket order (y zeroed), gate/up + swiglu, down + scatter.
int packed_prefill_impl(const moe_packed_layer_t& P, const float* x, int T, void* workspace, size_t workspace_bytes,
                        float* y, int32_t* ids_out, float* weights_out, cudaStream_t stream) {
  if (P.D > 4096 || P.F > 4096) return MOE_EUNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && y && workspace && P.w_router && P.g_qs && P.g_sf && P.u_qs && P.u_sf && P.d_qs && P.d_sf);
  MOE_REQUIRE(aligned(x, 16) && aligned(y, 16) && aligned(P.w_router, 16) && aligned(workspace, 256));
  MOE_REQUIRE(aligned(P.g_qs, 32) && aligned(P.u_qs, 32) && aligned(P.d_qs, 32));
  MOE_REQUIRE(aligned(P.g_sf, 16) && aligned(P.u_sf, 16) && aligned(P.d_sf, 16));
  MOE_REQUIRE(workspace_bytes >= layout_packed_prefill_workspace(T, P.D, P.F, P.k, P.E, nullptr, nullptr));
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  PackedPrefillWorkspace ws;
  layout_packed_prefill_workspace(T, P.D, P.F, P.k, P.E, static_cast<char*>(workspace), &ws);
  int32_t* ids = ids_out ? ids_out : ws.ids;
  float* wts = weights_out ? weights_out : ws.w;
  Launch L{stream, false};
  if ((rc = cuda_status(launch_route_topk(x, T, P.D, P.w_router, P.b_router, P.E, P.k, ws.logits, ws.rpart, ids, wts,
                                          L))) != MOE_OK)
    return rc;
  L.pdl = true;
  if ((rc = cuda_status(launch_bucket(ids, T, P.k, P.E, MOE_MM_TILE, (int)ws.max_rows, ws.counts, ws.basep, ws.rows,
                                      ws.inv, d->status, L))) != MOE_OK)
    return rc;
  if ((rc = cuda_status(launch_quant_rows_e2m1(x, T, P.D, P.k, ws.rows, ws.inv, ws.counts, ws.basep, P.E, (int)ws.max_rows, ws.aq,
                                               ws.asf, nullptr, ws.segs, ws.ctr, d->status, L))) != MOE_OK)
    return rc;
  GroupedMX4Args g{};
  g.kind = 0;
  g.w_qs[0] = P.g_qs;
  g.w_qs[1] = P.u_qs;
  g.w_sf[0] = P.g_sf;
  g.w_sf[1] = P.u_sf;
  g.bias[0] = P.bg;
  g.bias[1] = P.bu;
  g.E = P.E;
  g.R = P.F;
  g.C = P.D;
  g.counts = ws.counts;
  g.basep = ws.basep;
  g.rows = ws.rows;
  g.segs = ws.segs;
  g.ctr = ws.ctr;
  g.max_rows = (int)ws.max_rows;
  g.k = P.k;
  g.weights = wts;
  g.aq = ws.aq;
  g.asf = ws.asf;
  g.hf = ws.hf;
  g.alpha = 1.702f;
  g.limit = 7.0f;
  g.status = d->status;
  g.y = y;  // zeroed by the gate/up kernel, accumulated into by the down kernel
  g.ny = (int64_t)T * P.D;
  if ((rc = cuda_status(launch_grouped_mx4(g, L))) != MOE_OK) return rc;
  GroupedMX4Args gd = g;
  gd.kind = 1;
  gd.w_qs[0] = gd.w_qs[1] = P.d_qs;
  gd.w_sf[0] = gd.w_sf[1] = P.d_sf;
  gd.bias[0] = P.bd;
  gd.bias[1] = nullptr;
  gd.R = P.D;
  gd.C = P.F;
  if ((rc = cuda_status(launch_quant_h_e2m1(ws.hf, P.F, ws.rows, ws.counts, ws.basep, P.E, (int)ws.max_rows, ws.hq,
                                            ws.hsf, d->status, L))) != MOE_OK)
    return rc;
  gd.ctr = ws.ctr + 1;
  gd.aq = ws.hq;
  gd.asf = ws.hsf;
  gd.hf = nullptr;
  gd.y = y;
  return cuda_status(launch_grouped_mx4(gd, L));
}

int packed_layer_impl(const moe_packed_layer_t* Lp, const float* x, int T, int rail, void* workspace,
                      size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out, float* h_out,
                      cudaStream_t stream, int stages = MOE_STAGE_PROLOGUE | MOE_STAGE_GATEUP | MOE_STAGE_DOWN) {
  MOE_REQUIRE(Lp != nullptr && T >= 0);
  const moe_packed_layer_t& P = *Lp;
  MOE_REQUIRE(P.D >= 64 && P.F >= 64 && P.D % 64 == 0 && P.F % 64 == 0);
  MOE_REQUIRE(P.E >= 1 && P.E <= 256 && P.k >= 1 && P.k <= P.E && P.k <= 32);
  rail = resolve_packed_rail(T, rail);
  MOE_REQUIRE(rail == MOE_RAIL_DECODE_MX || rail == MOE_RAIL_GROUPED_MX || rail == MOE_RAIL_GROUPED_MX4);
  if (rail == MOE_RAIL_GROUPED_MX4) return packed_prefill_impl(P, x, T, workspace, workspace_bytes, y, ids_out,
                                                               weights_out, stream);
  if (rail != MOE_RAIL_DECODE_MX || T > MOE_GEMV_MAX_T) return MOE_EUNSUPPORTED;
  MOE_REQUIRE(T * P.k <= 64);
  if (P.D > 4096 || P.F > 4096) return MOE_EUNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(stages >= 1 && stages <= 7);
  MOE_REQUIRE(workspace && P.w_router && P.g_qs && P.g_sf && P.u_qs && P.u_sf && P.d_qs && P.d_sf);
  MOE_REQUIRE(x || !(stages & MOE_STAGE_PROLOGUE));
  MOE_REQUIRE(y || !(stages & MOE_STAGE_DOWN));
  MOE_REQUIRE(aligned(x, 16) && aligned(P.w_router, 16) && aligned(workspace, 256));
  MOE_REQUIRE(aligned(P.g_qs, 32) && aligned(P.u_qs, 32) && aligned(P.d_qs, 32));
  MOE_REQUIRE(aligned(P.g_sf, 16) && aligned(P.u_sf, 16) && aligned(P.d_sf, 16));
  const size_t need = layout_packed_workspace(T, P.D, P.F, P.k, P.E, nullptr, nullptr);
  MOE_REQUIRE(workspace_bytes >= need);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  PackedWorkspace ws;
  layout_packed_workspace(T, P.D, P.F, P.k, P.E, static_cast<char*>(workspace), &ws);
  const int npad = dmx::npad_for(T);
  Launch L{stream, false};
  if (stages & MOE_STAGE_PROLOGUE) {
    rc = cuda_status(launch_decode_prologue(x, T, P.D, P.w_router, P.b_router, P.E, ws.logits, ws.xq, ws.xsf,
                                            npad, ws.cnt, ws.ncnt, L));
    if (rc != MOE_OK) return rc;
  }
  L.pdl = true;
  DecodeMXArgs g{};
  g.kind = 0;
  g.w_qs[0] = P.g_qs;
  g.w_qs[1] = P.u_qs;
  g.w_sf[0] = P.g_sf;
  g.w_sf[1] = P.u_sf;
  g.bias[0] = P.bg;
  g.bias[1] = P.bu;
  g.E = P.E;
  g.R = P.F;
  g.C = P.D;
  g.T = T;
  g.k = P.k;
  g.b_q = ws.xq;
  g.b_sf = ws.xsf;
  g.logits = ws.logits;
  g.ids_out = ids_out;
  g.w_out = weights_out;
  g.alpha = 1.702f;
  g.limit = 7.0f;
  g.hq = ws.hq;
  g.hsf = ws.hsf;
  g.h_out = h_out;
  g.part = ws.part;
  g.cnt = ws.cnt;
  g.status = d->status;
  if (stages & MOE_STAGE_GATEUP) {
    rc = cuda_status(launch_decode_mx(g, L));
    if (rc != MOE_OK) return rc;
  }
  if (!(stages & MOE_STAGE_DOWN)) return MOE_OK;
  DecodeMXArgs dn{};
  dn.kind = 1;
  dn.w_qs[0] = dn.w_qs[1] = P.d_qs;
  dn.w_sf[0] = dn.w_sf[1] = P.d_sf;
  dn.bias[0] = P.bd;
  dn.E = P.E;
  dn.R = P.D;
  dn.C = P.F;
  dn.T = T;
  dn.k = P.k;
  dn.b_q = ws.hq;
  dn.b_sf = ws.hsf;
  dn.logits = ws.logits;
  dn.y = y;
  dn.part = ws.part;
  dn.cnt = ws.cnt + ws.ncnt_gu;
  dn.status = d->status;
  return cuda_status(launch_decode_mx(dn, L));
}
}  // namespace

extern "C" {

int moe_ffn_layer_packed(const moe_packed_layer_t* layer, const float* x, int T, int rail, void* workspace,
                         size_t workspace_bytes, float* y, int32_t* ids_out, float* weights_out, float* h_out,
                         cudaStream_t stream) {
  return packed_layer_impl(layer, x, T, rail, workspace, workspace_bytes, y, ids_out, weights_out, h_out, stream);
}

int moe_ffn_layer_packed_stage(const moe_packed_layer_t* layer, const float* x, int T, void* workspace,
                               size_t workspace_bytes, int stages, float* y, int32_t* ids_out,
                               float* weights_out, float* h_out, cudaStream_t stream) {
  return packed_layer_impl(layer, x, T, MOE_RAIL_DECODE_MX, workspace, workspace_bytes, y, ids_out, weights_out,
                           h_out, stream, stages);
}

int moe_ffn_layer_packed_hostio(const moe_packed_layer_t* layer, int T, int rail, void* workspace,
                                size_t workspace_bytes, const float* x_host, float* y_host, cudaStream_t stream) {
  MOE_REQUIRE(layer != nullptr && T >= 0);
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x_host && y_host && workspace && layer->D >= 64);
  const float* dx = static_cast<const float*>(mapped_host(x_host));
  float* dy = static_cast<float*>(const_cast<void*>(mapped_host(y_host)));
  if (dx && dy && aligned(dx, 16))  // pinned: the kernels read x and write y through the mapping
    return packed_layer_impl(layer, dx, T, rail, workspace, workspace_bytes, dy, nullptr, nullptr, nullptr, stream);
  const int prail = resolve_packed_rail(T, rail);
  float* xs = nullptr;
  float* ys = nullptr;
  MOE_REQUIRE(aligned(workspace, 256));
  if (prail == MOE_RAIL_GROUPED_MX4) {
    MOE_REQUIRE(workspace_bytes >=
                layout_packed_prefill_workspace(T, layer->D, layer->F, layer->k, layer->E, nullptr, nullptr));
    PackedPrefillWorkspace pw;
    layout_packed_prefill_workspace(T, layer->D, layer->F, layer->k, layer->E, static_cast<char*>(workspace), &pw);
    xs = pw.xs;
    ys = pw.ys;
  } else {
    if (prail != MOE_RAIL_DECODE_MX || T > MOE_GEMV_MAX_T) return MOE_EUNSUPPORTED;
    MOE_REQUIRE(workspace_bytes >=
                layout_packed_workspace(T, layer->D, layer->F, layer->k, layer->E, nullptr, nullptr));
    PackedWorkspace ws;
    layout_packed_workspace(T, layer->D, layer->F, layer->k, layer->E, static_cast<char*>(workspace), &ws);
    xs = ws.xs;
    ys = ws.ys;
  }
  const size_t bytes = (size_t)T * layer->D * sizeof(float);
  cudaError_t err = cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, stream);
  if (err != cudaSuccess) return cuda_status(err);
  const int rc = packed_layer_impl(layer, xs, T, rail, workspace, workspace_bytes, ys, nullptr, nullptr, nullptr,
                                   stream);
  if (rc != MOE_OK) return rc;
  return cuda_status(cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, stream));
}

int moe_checked_build(void) {
#ifdef MOE_CHECKED
  return 1;
#else
  return 0;
#endif
}

int moe_get_status(cudaStream_t stream, int* status) {
  MOE_REQUIRE(status != nullptr);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return cuda_status(err);
  int v = 0;
  if ((err = cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_status(err);
  const int zero = 0;
  if ((err = cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_status(err);
  *status = v;
  return MOE_OK;
}

int moe_get_timeout_site(cudaStream_t stream, int* site) {
  MOE_REQUIRE(site != nullptr);
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != MOE_OK) return rc;
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return cuda_status(err);
  int v = 0;
  if ((err = cudaMemcpy(&v, d->status + 1, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_status(err);
  const int zero = 0;
  if ((err = cudaMemcpy(d->status + 1, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_status(err);
  *site = v;
  return MOE_OK;
}

int moe_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
