// C ABI entry points that are not tied to one kernel: argument checks, the
// choice between the decode and the prefill kernel, status strings and the
// device error word.
#include <cstdint>
#include <mutex>

#include "decode_group.h"
#include "tm_common.cuh"

namespace w4 {

namespace {
thread_local int t_launches = 0;
std::mutex g_mu;
int g_sms[64] = {0};
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;
}  // namespace

EncodeTiledFn encode_tiled_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

int num_sms(int device) {
  if (device < 0 || device >= 64) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[device]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0) v = 148;
    g_sms[device] = v;
  }
  return g_sms[device];
}

void sm_shared_memory(int device, int* per_sm, int* reserved_per_cta) {
  static int cache[64][2];
  if (device < 0 || device >= 64) {
    *per_sm = 228 * 1024;
    *reserved_per_cta = 1024;
    return;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!cache[device][0]) {
    int a = 0, b = 0;
    if (cudaDeviceGetAttribute(&a, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess || a <= 0)
      a = 228 * 1024;
    if (cudaDeviceGetAttribute(&b, cudaDevAttrReservedSharedMemoryPerBlock, device) != cudaSuccess || b < 0)
      b = 1024;
    cache[device][0] = a;
    cache[device][1] = b;
  }
  *per_sm = cache[device][0];
  *reserved_per_cta = cache[device][1];
}

void set_launch_count(int n) { t_launches = n; }

int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess ? d : 0;
}

// Largest M the decode kernel serves, and the largest it gets when the path
// is automatic; above that the tensor-memory kernel runs (measured faster on
// GB300 from M = 33 up).
constexpr int kDecodeMaxM = 64;
constexpr int kAutoDecodeMaxM = 32;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static tm_status plan(const tm_packed* p, int M, const tm_gemm_config* cfg, tm_gemm_config* out) {
  int path = cfg ? cfg->path : 0;
  if (path == 0) path = M <= kAutoDecodeMaxM ? 1 : 3;
  if (path == 1) {
    if (M > kDecodeMaxM) return TM_ERR_UNSUPPORTED;
    return plan_decode(p, M, cfg, out);
  }
  if (path == 2) return plan_prefill(p, M, cfg, out);
  if (path == 3) return plan_tc(p, M, cfg, out);
  return TM_ERR_INVALID_ARG;
}

// Sticky error bits of the KV-cache kernels (kv.cu) and the W8A8 GEMM (w8a8.cu).
cudaError_t kv_error_bits(uint32_t* bits, bool clear);
cudaError_t w8_error_bits(uint32_t* bits, bool clear);
cudaError_t rtn_error_bits(uint32_t* bits, bool clear);

// Self-test of the bounded barrier wait every kernel uses: one warp waits on
// an mbarrier that nothing ever arrives on; after kWaitLimitNs it must give
// up, raise the abort flag and set the timeout bit, and the kernel returns.
static __device__ uint32_t s_err_selftest;

__global__ void wait_timeout_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, reinterpret_cast<volatile int*>(&abort_flag), &s_err_selftest);
}

}  // namespace w4

using namespace w4;

extern "C" tm_status tm_selftest_wait_timeout(void* stream) {
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

extern "C" const char* tm_status_str(tm_status s) {
  switch (s) {
    case TM_OK: return "ok";
    case TM_ERR_INVALID_ARG: return "invalid argument";
    case TM_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case TM_ERR_UNSUPPORTED: return "unsupported configuration";
    case TM_ERR_CUDA: return "CUDA call failed";
    case TM_ERR_DEVICE_TIMEOUT: return "device barrier timeout";
    case TM_ERR_BAD_CODE: return "code or zero above 15";
    case TM_ERR_SCRATCH_LIMIT: return "request exceeds the static staging array";
  }
  return "unknown status";
}

extern "C" tm_status tm_gemm_plan(const tm_packed* p, int M, const tm_gemm_config* cfg, tm_gemm_config* out) {
  if (!p || !out || M < 0) return TM_ERR_INVALID_ARG;
  return plan(p, M > 0 ? M : 1, cfg, out);
}

extern "C" tm_status tm_w4a16_gemm_ex(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config* cfg,
                                      void* stream) {
  t_launches = 0;
  if (!p || M < 0) return TM_ERR_INVALID_ARG;
  if (M == 0) return TM_OK;
  if (!X || !Y) return TM_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Y)) return TM_ERR_ALIGNMENT;
  tm_gemm_config c;
  tm_status st = plan(p, M, cfg, &c);
  if (st != TM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (c.path == 1) return launch_decode(X, p, Y, M, c, s);
  if (c.path == 3) return launch_tc(X, p, Y, M, c, s);
  return launch_prefill(X, p, Y, M, c, s);
}

extern "C" tm_status tm_w4a16_gemm_silu_mul(const void* X, const tm_packed* p, void* H, int M,
                                            const tm_gemm_config* cfg, void* stream) {
  t_launches = 0;
  if (!p || M < 0) return TM_ERR_INVALID_ARG;
  if (p->L.N % 8 != 0) return TM_ERR_INVALID_ARG;
  if (M == 0) return TM_OK;
  if (!X || !H) return TM_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(H)) return TM_ERR_ALIGNMENT;
  tm_gemm_config c;
  tm_status st = plan(p, M, cfg, &c);
  if (st != TM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (c.path == 1) return launch_decode(X, p, H, M, c, s, true);
  if (c.path == 3) return launch_tc(X, p, H, M, c, s, true);
  return TM_ERR_UNSUPPORTED;  // the shared-memory prefill kernel has no fused epilogue
}

extern "C" tm_status tm_w4a16_gemm(const void* X, const tm_packed* p, void* Y, int M, void* stream) {
  return tm_w4a16_gemm_ex(X, p, Y, M, nullptr, stream);
}

namespace {

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Checks of tm_w4a16_gemm_grouped's arguments; on TM_OK fills jobs and ps.
tm_status check_group(const tm_gemm_problem* probs, int n, int M, DecodeJob* jobs, const tm_packed** ps) {
  if (!probs || n < 1 || n > TM_GROUP_MAX || M < 0) return TM_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const tm_gemm_problem& q = probs[i];
    if (!q.p || (M > 0 && (!q.X || !q.Y))) return TM_ERR_INVALID_ARG;
    if (q.p->L.g != probs[0].p->L.g || q.p->device != probs[0].p->device) return TM_ERR_INVALID_ARG;
    if (q.silu && q.p->L.N % 8 != 0) return TM_ERR_INVALID_ARG;
    jobs[i] = {q.X, q.p, q.Y, q.silu != 0};
    ps[i] = q.p;
  }
  if (M == 0) return TM_OK;
  for (int i = 0; i < n; ++i) {
    if (!aligned16(probs[i].X) || !aligned16(probs[i].Y)) return TM_ERR_ALIGNMENT;
    const size_t yb = (size_t)M * (probs[i].silu ? probs[i].p->L.N / 2 : probs[i].p->L.N) * 2;
    for (int j = 0; j < n; ++j) {
      const size_t xb = (size_t)M * probs[j].p->L.K * 2;
      if (ranges_overlap(probs[i].Y, yb, probs[j].X, xb)) return TM_ERR_INVALID_ARG;
      if (j != i) {
        const size_t yb2 = (size_t)M * (probs[j].silu ? probs[j].p->L.N / 2 : probs[j].p->L.N) * 2;
        if (ranges_overlap(probs[i].Y, yb, probs[j].Y, yb2)) return TM_ERR_INVALID_ARG;
      }
    }
  }
  return TM_OK;
}

// Grouped launch when the path is the decode kernel (explicit path 1, or
// automatic with M <= 32); *grouped = false means one launch per product.
tm_status plan_group(const tm_packed* const* ps, int n, int M, const tm_gemm_config* cfg, tm_gemm_config* out,
                     int* splits, bool* grouped) {
  const int path = cfg ? cfg->path : 0;
  if (path != 0 && path != 1) return TM_ERR_INVALID_ARG;
  *grouped = path == 1 || M <= kAutoDecodeMaxM;
  if (!*grouped) return TM_OK;
  if (M > kDecodeMaxM) return TM_ERR_UNSUPPORTED;
  return plan_decode_group(ps, n, M > 0 ? M : 1, cfg, out, splits);
}

}  // namespace

extern "C" tm_status tm_gemm_plan_grouped(const tm_gemm_problem* probs, int n, int M, const tm_gemm_config* cfg,
                                          tm_gemm_config* out, int* splits) {
  DecodeJob jobs[TM_GROUP_MAX];
  const tm_packed* ps[TM_GROUP_MAX];
  if (!out) return TM_ERR_INVALID_ARG;
  tm_status st = check_group(probs, n, 0, jobs, ps);
  if (st != TM_OK) return st;
  bool grouped = false;
  st = plan_group(ps, n, M, cfg, out, splits, &grouped);
  if (st != TM_OK || grouped) return st;
  // One launch per product: each product's own automatic settings.
  for (int i = n - 1; i >= 0; --i) {
    st = plan(ps[i], M, nullptr, out);
    if (st != TM_OK) return st;
    if (splits) splits[i] = out->split_k;
  }
  return TM_OK;
}

extern "C" tm_status tm_w4a16_gemm_grouped(const tm_gemm_problem* probs, int n, int M, const tm_gemm_config* cfg,
                                           void* stream) {
  t_launches = 0;
  DecodeJob jobs[TM_GROUP_MAX];
  const tm_packed* ps[TM_GROUP_MAX];
  tm_status st = check_group(probs, n, M, jobs, ps);
  if (st != TM_OK || M == 0) return st;
  tm_gemm_config c;
  bool grouped = false;
  st = plan_group(ps, n, M, cfg, &c, nullptr, &grouped);
  if (st != TM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (grouped) return launch_decode_group(jobs, n, M, cfg, s);
  // Every product is planned before the first launch.
  tm_gemm_config cs[TM_GROUP_MAX];
  for (int i = 0; i < n; ++i) {
    st = plan(ps[i], M, nullptr, &cs[i]);
    if (st != TM_OK) return st;
  }
  int launches = 0;
  for (int i = 0; i < n; ++i) {
    st = probs[i].silu ? tm_w4a16_gemm_silu_mul(probs[i].X, ps[i], probs[i].Y, M, &cs[i], stream)
                       : tm_w4a16_gemm_ex(probs[i].X, ps[i], probs[i].Y, M, &cs[i], stream);
    if (st != TM_OK) return st;
    launches += t_launches;
  }
  t_launches = launches;
  return TM_OK;
}

extern "C" tm_status tm_w4a16_gemm_host(const void* X_host, const tm_packed* p, void* Y_host, int M, void* X_dev,
                                        void* Y_dev, const tm_gemm_config* cfg, void* stream) {
  t_launches = 0;
  if (!p || M < 0) return TM_ERR_INVALID_ARG;
  if (M == 0) return TM_OK;
  if (!X_host || !Y_host || !X_dev || !Y_dev) return TM_ERR_INVALID_ARG;
  if (!aligned16(X_dev) || !aligned16(Y_dev)) return TM_ERR_ALIGNMENT;
  tm_gemm_config c;
  tm_status st = plan(p, M, cfg, &c);  // reject before touching any buffer
  if (st != TM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)M * p->L.K * 2, yb = (size_t)M * p->L.N * 2;
  if (cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return TM_ERR_CUDA;
  st = tm_w4a16_gemm_ex(X_dev, p, Y_dev, M, &c, s);
  if (st != TM_OK) return st;
  return cudaMemcpyAsync(Y_host, Y_dev, yb, cudaMemcpyDeviceToHost, s) == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

extern "C" tm_status tm_w4a16_gemm_host_batch(int n, const tm_packed* const* p, const int* M, const void* X_host,
                                              void* Y_host, void* X_dev, void* Y_dev, void* stream) {
  t_launches = 0;
  if (n < 0 || (n > 0 && (!p || !M))) return TM_ERR_INVALID_ARG;
  size_t xb = 0, yb = 0;
  for (int i = 0; i < n; ++i) {
    if (!p[i] || M[i] < 0) return TM_ERR_INVALID_ARG;
    if (M[i] == 0) continue;
    tm_gemm_config c;
    const tm_status st = plan(p[i], M[i], nullptr, &c);  // reject before touching any buffer
    if (st != TM_OK) return st;
    xb += (size_t)M[i] * p[i]->L.K * 2;
    yb += (size_t)M[i] * p[i]->L.N * 2;
  }
  if (xb == 0) return TM_OK;
  if (!X_host || !Y_host || !X_dev || !Y_dev) return TM_ERR_INVALID_ARG;
  if (!aligned16(X_dev) || !aligned16(Y_dev)) return TM_ERR_ALIGNMENT;
  // Runs of consecutive products with the same M <= 32 and group size (at
  // most TM_GROUP_MAX) share one grouped launch: their staging regions are
  // disjoint, so the products are independent.
  auto run_end = [&](int i) {
    int j = i + 1;
    if (M[i] > kAutoDecodeMaxM) return j;
    while (j < n && j - i < TM_GROUP_MAX && M[j] == M[i] && p[j]->L.g == p[i]->L.g && p[j]->device == p[i]->device)
      ++j;
    return j;
  };
  for (int i = 0; i < n;) {
    const int j = M[i] > 0 ? run_end(i) : i + 1;
    if (j - i > 1) {
      tm_gemm_config c;
      const tm_status st = plan_decode_group(p + i, j - i, M[i], nullptr, &c, nullptr);
      if (st != TM_OK) return st;
    }
    i = j;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return TM_ERR_CUDA;
  size_t xo = 0, yo = 0;
  int launches = 0;
  for (int i = 0; i < n;) {
    if (M[i] == 0) {
      ++i;
      continue;
    }
    const int j = run_end(i);
    DecodeJob jobs[TM_GROUP_MAX];
    for (int k = i; k < j; ++k) {
      jobs[k - i] = {static_cast<const char*>(X_dev) + xo, p[k], static_cast<char*>(Y_dev) + yo, false};
      xo += (size_t)M[k] * p[k]->L.K * 2;
      yo += (size_t)M[k] * p[k]->L.N * 2;
    }
    const tm_status st = j - i > 1 ? launch_decode_group(jobs, j - i, M[i], nullptr, s)
                                   : tm_w4a16_gemm_ex(jobs[0].X, p[i], jobs[0].Y, M[i], nullptr, stream);
    if (st != TM_OK) return st;
    launches += t_launches;
    i = j;
  }
  if (cudaMemcpyAsync(Y_host, Y_dev, yb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return TM_ERR_CUDA;
  t_launches = launches;
  return TM_OK;
}

extern "C" tm_status tm_device_error(int clear, uint32_t* bits) {
  if (cudaDeviceSynchronize() != cudaSuccess) return TM_ERR_CUDA;
  uint32_t a = 0, b = 0, c = 0, d = 0, e = 0, f = 0, h = 0, r = 0;
  if (pack_error_bits(&a, clear != 0) != cudaSuccess || decode_error_bits(&b, clear != 0) != cudaSuccess ||
      prefill_error_bits(&c, clear != 0) != cudaSuccess || tc_error_bits(&d, clear != 0) != cudaSuccess ||
      kv_error_bits(&f, clear != 0) != cudaSuccess || w8_error_bits(&h, clear != 0) != cudaSuccess ||
      rtn_error_bits(&r, clear != 0) != cudaSuccess ||
      cudaMemcpyFromSymbol(&e, s_err_selftest, sizeof(e)) != cudaSuccess)
    return TM_ERR_CUDA;
  if (clear && e) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(s_err_selftest, &zero, sizeof(zero)) != cudaSuccess) return TM_ERR_CUDA;
  }
  const uint32_t v = (a | b | c | d | e | f | h | r) & kErrTimeout;
  if (bits) *bits = v;
  return v ? TM_ERR_DEVICE_TIMEOUT : TM_OK;
}

extern "C" int tm_last_launch_count(void) { return t_launches; }
