// Shared pieces of the CUDA path: the packed-weight layout, the handle, and
// thin inline-PTX wrappers for mbarriers, bulk/TMA copies, tcgen05 and clusters
// on sm_103a.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tm_w4a16.h"

// ---------------------------------------------------------------------------
// Packed layout (ours; the pages fix only "fragments in MMA lane order").
//
// A unit is 16 columns (an n-tile) x 64 k = 1024 codes = 512 bytes, stored as
// 32 lanes x 16 bytes.  Lane l = 4*gr + t holds rows (n0+gr, n0+gr+8) and
// k = k0 + 16t .. 16t+15 as four 32-bit words; word `st` holds k = 16t+4st+j,
// j = 0..3, for the two rows.  Nibble i of a word (bits 4i..4i+3):
//   row  = gr + 8*(i & 1)
//   j    = 2*((i >> 1) & 1) + (i >> 2)
// so (w & 0x000F000F) gives row gr at k, k+1; (w & 0x00F000F0) row gr+8 at
// k, k+1; the same on w >> 8 gives k+2, k+3.  One word is exactly one
// mma.m16n8k16 A fragment of W^T (rows = n, columns = k) once the k order of
// the step is permuted the same way on X (slot 2t -> 4t, 2t+1 -> 4t+1,
// 2t+8 -> 4t+2, 2t+9 -> 4t+3).
//
// Regions (one allocation, each 1024-byte aligned), ordered by pairs of groups
// ("super-groups", SG = 2g values of k) first, so that the codes, scales and
// zeros one CTA needs for one super-group of consecutive n-tiles are each a
// single contiguous run:
//   codes  [NSG][NT][UPS][512 B]     UPS = 2g/64 units per super-group
//   scales [NSG][NT][2][16 x fp16]   element 2*gr + h = s[grp][n0 + gr + 8h]
//   zeros  [NSG][NT][16 B]           byte (grp&1)*8 + gr: low nibble z of row gr,
//                                    high nibble z of row gr+8
// NT = N/16; NSG = Kp/(2g), with Kp = K rounded up to 2g; the padding group
// holds zero codes, zeros and scales.
// ---------------------------------------------------------------------------

namespace w4 {

constexpr int kUnitK = 64;
constexpr int kUnitBytes = 512;

struct Layout {
  int K, N, g;
  int Kp, NT, KT, G, NSG, UPS;
  size_t codes_off, scales_off, zeros_off, total;
};

inline Layout make_layout(int K, int N, int g) {
  Layout L;
  L.K = K;
  L.N = N;
  L.g = g;
  L.Kp = ((K + 2 * g - 1) / (2 * g)) * (2 * g);
  L.NT = N / 16;
  L.KT = L.Kp / kUnitK;
  L.G = L.Kp / g;
  L.NSG = L.G / 2;
  L.UPS = 2 * g / kUnitK;
  auto al = [](size_t v) { return (v + 1023) & ~size_t(1023); };
  L.codes_off = 0;
  size_t codes = (size_t)L.NT * L.KT * kUnitBytes;
  L.scales_off = al(codes);
  size_t scales = (size_t)L.NT * L.G * 32;
  L.zeros_off = al(L.scales_off + scales);
  size_t zeros = (size_t)L.NT * L.NSG * 16;
  L.total = al(L.zeros_off + zeros);
  return L;
}

}  // namespace w4

struct tm_packed {
  w4::Layout L;
  int device;
  uint8_t* base;  // device allocation
  // TMA descriptors over the packed regions (prefill kernel: 16 n-tiles a box)
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  CUtensorMap tm_zeros;
  // The same for the tensor-memory kernel: 8 n-tiles a box, codes as 128-byte
  // rows with the 128-byte swizzle (a conflict-free transposed read)
  CUtensorMap tc_codes;
  CUtensorMap tc_scales;
  CUtensorMap tc_zeros;
};

namespace w4 {

// w / s for the quantisers' rounding rule, q = rint(w / s), from the
// reciprocal i = fl(1/s) computed once per scale: t = w i, the remainder
// w - t s by one fma, and one correction t + (w - t s) i by another.  For fp16
// w and s (the weight and KV quantisers) rint of the result equals rint of the
// exact quotient: at a half-integer quotient h the correction lands on h
// itself (the remaining error is below 2^-46 h), and any other quotient of two
// fp16 values lies at least 1/8188 from every half-integer, far more than the
// result's error of about one binary32 ulp.  w * i alone can miss an exact
// tie by an ulp and round it the wrong way.
__device__ __forceinline__ float fp16_quotient(float w, float s, float i) {
  const float t = __fmul_rn(w, i);
  const float r = __fmaf_rn(-t, s, w);
  return __fmaf_rn(r, i, t);
}

// Device-side sticky error bits (per device; read by tm_device_error).
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBadCode = 2u;

// Barrier waits give up after this long (a normal wait lasts microseconds).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Driver entry point for tensor-map encoding (no link against libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Sticky device error bits of each translation unit (read, optionally cleared;
// synchronises the device).
cudaError_t pack_error_bits(uint32_t* bits, bool clear);
cudaError_t decode_error_bits(uint32_t* bits, bool clear);
cudaError_t prefill_error_bits(uint32_t* bits, bool clear);
cudaError_t tc_error_bits(uint32_t* bits, bool clear);

// Common host launch helpers (defined in api.cu).
int num_sms(int device);
// Shared memory of one SM that resident CTAs share, and the part of it the
// system reserves for each CTA (bytes).
void sm_shared_memory(int device, int* per_sm, int* reserved_per_cta);
void set_launch_count(int n);
// The device current on this thread (0 when the query fails).
int current_device();

// The dynamic shared-memory limit of a kernel is a per-device setting: raise
// it once per (kernel, device).  `done` is the kernel's own flag word (bit d =
// device d); two threads making their first call at once may both set it,
// which is harmless.
inline bool smem_attr_once(std::atomic<unsigned long long>& done, const void* kern, int bytes) {
  const int dev = current_device();
  const unsigned long long bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

// Decode / prefill launchers (decode.cu, prefill.cu).
tm_status plan_decode(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out);
tm_status launch_decode(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& cfg,
                        cudaStream_t stream, bool silu = false);
tm_status plan_prefill(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out);
tm_status launch_prefill(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& cfg,
                         cudaStream_t stream);
tm_status plan_tc(const tm_packed* p, int M, const tm_gemm_config* in, tm_gemm_config* out);
tm_status launch_tc(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config& cfg,
                    cudaStream_t stream, bool silu = false);

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One try: the hardware may suspend the thread for a system-dependent time
// while the phase is incomplete (measured on GB300: an explicit suspend-time
// hint was no faster, and 3% slower in the tensor-memory kernel).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase with `parity` completed; false when the
// block-wide abort flag is raised or the wait exceeded kWaitLimitNs (which
// raises the flag and the device error bit).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte multiples).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load, completing on an mbarrier.  x (innermost) must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
      "%6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

template <uint32_t LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Four 16-bit halves pairs (q - z) from one packed word, exact in fp16.
//   zz_lo = (1024 + z_row_gr) twice; zf_hi = -(64 + z_row_gr8) twice.
// 0x6400 is 1024.0 in fp16: OR-ing a nibble into its low mantissa bits gives
// 1024 + q; OR-ing a nibble shifted by 4 gives 1024 + 16 q.
//   out[0] = row gr  , k, k+1      out[1] = row gr+8, k, k+1
//   out[2] = row gr  , k+2, k+3    out[3] = row gr+8, k+2, k+3
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t zz_lo, uint32_t zf_hi, uint32_t out[4]) {
  constexpr uint32_t kMagic = 0x64006400u;
  constexpr uint32_t kSixteenth = 0x2C002C00u;  // 1/16 in both halves
  const uint32_t w8 = w >> 8;
  const uint32_t r0 = lop3<0xEA>(w, 0x000F000Fu, kMagic);   // (a & b) | c
  const uint32_t r1 = lop3<0xEA>(w, 0x00F000F0u, kMagic);
  const uint32_t r2 = lop3<0xEA>(w8, 0x000F000Fu, kMagic);
  const uint32_t r3 = lop3<0xEA>(w8, 0x00F000F0u, kMagic);
  out[0] = hsub2_u32(r0, zz_lo);
  out[1] = hfma2_u32(r1, kSixteenth, zf_hi);
  out[2] = hsub2_u32(r2, zz_lo);
  out[3] = hfma2_u32(r3, kSixteenth, zf_hi);
}

// The raw form: the four A-fragment registers of a word without the zero
// point, 5 instructions per 8 weights.
//   out[0] = 1024 + q (row gr  , k, k+1)     out[1] = 1024 + 16 q (row gr+8, k, k+1)
//   out[2] = 1024 + q (row gr  , k+2, k+3)   out[3] = 1024 + 16 q (row gr+8, k+2, k+3)
// A product with these sums x (1024 + q) (resp. x (1024 + 16 q)); the zero
// point and the offset are removed once per group with the sum of x.
__device__ __forceinline__ void raw_word(uint32_t w, uint32_t out[4]) {
  constexpr uint32_t kMagic = 0x64006400u;
  const uint32_t w8 = w >> 8;
  out[0] = lop3<0xEA>(w, 0x000F000Fu, kMagic);
  out[1] = lop3<0xEA>(w, 0x00F000F0u, kMagic);
  out[2] = lop3<0xEA>(w8, 0x000F000Fu, kMagic);
  out[3] = lop3<0xEA>(w8, 0x00F000F0u, kMagic);
}

// (1024 + z) in both halves of a word.
__device__ __forceinline__ uint32_t zero_pair_lo(uint32_t z) {
  const uint32_t h = 0x6400u | z;
  return h | (h << 16);
}
// -(64 + z) in both halves: 64 + z (z < 16) is 2^6 (1 + z/64), i.e. the fp16
// pattern 0x5400 + 16 z; the sign bit makes it 0xD400 + 16 z.
__device__ __forceinline__ uint32_t zero_pair_hi(uint32_t z) {
  const uint32_t b = 0xD400u + (z << 4);
  return b | (b << 16);
}

// d = a . b with a zero accumulator (no register moves to clear d).
__device__ __forceinline__ void mma_16816_zc(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Pure register operation (not volatile): the compiler may schedule it freely.
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---- clusters -------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split form: arrive early, wait before the first access to another CTA's
// shared memory (it must have started running).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---- programmatic dependent launch ------------------------------------------
// Wait until the preceding grid in the stream finished and its writes are
// visible (no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid in the stream to begin launching.
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// silu(gate) * up for the fused gate/up epilogue, in fp32 (expf and an IEEE
// division; silu(x) = x / (1 + exp(-x))).
__device__ __forceinline__ float silu_mul(float gate, float up) {
  return __fdiv_rn(gate, 1.f + expf(-gate)) * up;
}

// ---- tcgen05 --------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16, single CTA.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once all prior tcgen05 operations of this thread completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// The eight epilogue warps (2..9) of the tensor-memory kernels, on named
// barrier 1 (the TMA and MMA warps take no part).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// TMA tensor store of a 2-D box from shared memory, as a bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until the bulk groups have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] . B[smem desc]^T, kind::f16, single CTA.  A occupies
// tensor-memory lanes 0..127 (its rows) and 8 columns per 16 k (column c holds
// k = 2c in the low half and 2c + 1 in the high half).
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 lanes x 8 columns: lane (4 gr + t) stores r0, r1 into tensor-memory lane
// (base + gr) at columns 2t, 2t + 1 and r2, r3 into lane (base + gr + 8) at
// the same columns -- the mma.m16n8 accumulator layout.
__device__ __forceinline__ void tc_st_16x256b(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3));
}

// 32 lanes x 8 consecutive 32-bit columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tc_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);       // start address
  d |= (uint64_t)1u << 16;                       // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset: next 8-row atom
  d |= (uint64_t)1u << 46;                       // descriptor version for tcgen05
  d |= (uint64_t)2u << 61;                       // swizzle: 128B
  return d;
}

// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

#endif  // __CUDACC__

}  // namespace w4

