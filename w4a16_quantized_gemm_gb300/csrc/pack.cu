// Offline weight packing (the guide's section 1, "Hardware-Aware Weight
// Packing"): plain codes, zeros and scales in, the kernels' fragment order
// out, once per layer.  The pages' own packer widens codes to 16 bits and lets
// ldmatrix redistribute them across lanes; here the destination order is
// computed directly per output word (see tm_common.cuh for the layout), which
// needs no shared-memory staging and is trivially bit-exact to invert.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "tm_common.cuh"

namespace w4 {

static __device__ uint32_t s_err_pack;

// One thread per 32-bit code word.
// Word index = (((sg*NT + nt)*UPS + u)*32 + lane)*4 + st.
__global__ void pack_codes_kernel(const uint8_t* __restrict__ q, int K, int N, int NT, int UPS, long long nwords,
                                  uint32_t* __restrict__ out) {
  long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= nwords) return;
  const int st = (int)(w & 3);
  const int lane = (int)((w >> 2) & 31);
  const long long unit = w >> 7;
  const int u = (int)(unit % UPS);
  const long long rest = unit / UPS;
  const int nt = (int)(rest % NT);
  const int sg = (int)(rest / NT);
  const int kt = sg * UPS + u;
  const int gr = lane >> 2, t = lane & 3;
  uint32_t word = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = gr + 8 * (i & 1);
    const int j = 2 * ((i >> 1) & 1) + (i >> 2);
    const int n = nt * 16 + row;
    const int k = kt * kUnitK + 16 * t + 4 * st + j;
    uint32_t c = 0;
    if (n < N && k < K) {
      c = q[(size_t)k * N + n];
      if (c > 15) {
        bad = true;
        c &= 15;
      }
    }
    word |= c << (4 * i);
  }
  if (bad) atomicOr(&s_err_pack, kErrBadCode);
  out[w] = word;
}

// One thread per (sg, nt, group of the pair, gr): the fp16 pair (s[n0+gr], s[n0+gr+8]).
__global__ void pack_scales_kernel(const uint16_t* __restrict__ s, int Gk, int N, int NT, long long npairs,
                                   uint32_t* __restrict__ out) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= npairs) return;
  const int gr = (int)(i & 7);
  const int gi = (int)((i >> 3) & 1);
  const long long rest = i >> 4;
  const int nt = (int)(rest % NT);
  const int grp = 2 * (int)(rest / NT) + gi;
  uint32_t lo = 0, hi = 0;
  const int n = nt * 16 + gr;
  if (grp < Gk) {
    if (n < N) lo = s[(size_t)grp * N + n];
    if (n + 8 < N) hi = s[(size_t)grp * N + n + 8];
  }
  out[i] = lo | (hi << 16);
}

// One thread per zero byte: (sg, nt, byte b) -> group 2*sg + (b >> 3), row b & 7.
__global__ void pack_zeros_kernel(const uint8_t* __restrict__ z, int Gk, int N, int NT, long long nbytes,
                                  uint8_t* __restrict__ out) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nbytes) return;
  const int b = (int)(i & 15);
  const long long rest = i >> 4;
  const int nt = (int)(rest % NT);
  const int sg = (int)(rest / NT);
  const int grp = 2 * sg + (b >> 3);
  const int gr = b & 7;
  const int n = nt * 16 + gr;
  uint32_t lo = 0, hi = 0;
  if (grp < Gk) {
    if (n < N) lo = z[(size_t)grp * N + n];
    if (n + 8 < N) hi = z[(size_t)grp * N + n + 8];
  }
  if (lo > 15 || hi > 15) atomicOr(&s_err_pack, kErrBadCode);
  out[i] = (uint8_t)((lo & 15) | ((hi & 15) << 4));
}

// Inverse: one thread per (k, n) code.
__global__ void unpack_codes_kernel(const uint32_t* __restrict__ words, int K, int N, int NT, int UPS,
                                    uint8_t* __restrict__ q) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)K * N) return;
  const int k = (int)(i / N), n = (int)(i % N);
  const int nt = n >> 4, r = n & 15, gr = r & 7, hirow = r >> 3;
  const int kt = k / kUnitK, kk = k % kUnitK, t = kk >> 4, st = (kk >> 2) & 3, j = kk & 3;
  const int lane = gr * 4 + t;
  const int nib = hirow + 2 * (j >> 1) + 4 * (j & 1);
  const int sg = kt / UPS, u = kt % UPS;
  const uint32_t w = words[((((size_t)sg * NT + nt) * UPS + u) * 32 + lane) * 4 + st];
  q[i] = (uint8_t)((w >> (4 * nib)) & 15);
}

__global__ void unpack_meta_kernel(const uint16_t* __restrict__ sp, const uint8_t* __restrict__ zp, int Gk, int N,
                                   int NT, uint8_t* __restrict__ z, uint16_t* __restrict__ s) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)Gk * N) return;
  const int grp = (int)(i / N), n = (int)(i % N);
  const int nt = n >> 4, r = n & 15, gr = r & 7, hirow = r >> 3;
  const int sg = grp >> 1;
  s[i] = sp[(((size_t)sg * NT + nt) * 2 + (grp & 1)) * 16 + 2 * gr + hirow];
  const uint8_t b = zp[((size_t)sg * NT + nt) * 16 + (grp & 1) * 8 + gr];
  z[i] = hirow ? (b >> 4) : (b & 15);
}

cudaError_t pack_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_pack, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_pack, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

// Tensor map (swizzle none unless asked): dims[0] innermost, strides in bytes for dims 1..rank-1.
static bool encode_nd(CUtensorMap* map, CUtensorMapDataType dt, void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  CUresult r = fn(map, dt, (cuuint32_t)rank, base, d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static unsigned grid_for(long long n, int block) { return (unsigned)((n + block - 1) / block); }

static bool valid_shape(int K, int N, int g) {
  if (g != 64 && g != 128) return false;
  if (K <= 0 || N <= 0 || K % g != 0 || N % 16 != 0) return false;
  // keep every index of the packed buffer in 32-bit-safe ranges
  if ((long long)K * N > (1ll << 34)) return false;
  return true;
}

}  // namespace w4

using namespace w4;

extern "C" tm_status tm_packed_bytes(int K, int N, int g, size_t* bytes) {
  if (!bytes || !valid_shape(K, N, g)) return TM_ERR_INVALID_ARG;
  *bytes = make_layout(K, N, g).total;
  return TM_OK;
}

extern "C" tm_status tm_pack_weights(const uint8_t* q, const uint8_t* z, const uint16_t* s, int K, int N, int g,
                                     tm_packed** out) {
  if (!out) return TM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!q || !z || !s || !valid_shape(K, N, g)) return TM_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TM_ERR_CUDA;
  tm_packed* p = new (std::nothrow) tm_packed;
  if (!p) return TM_ERR_CUDA;
  memset(p, 0, sizeof(*p));
  p->L = make_layout(K, N, g);
  p->device = dev;
  const Layout& L = p->L;
  if (cudaMalloc(&p->base, L.total) != cudaSuccess) {
    delete p;
    return TM_ERR_CUDA;
  }
  uint32_t bits = 0;
  cudaError_t e = pack_error_bits(&bits, true);
  const int B = 256;
  const long long nwords = (long long)L.NT * L.KT * 128;
  const long long npairs = (long long)L.NT * L.G * 8;
  const long long nzb = (long long)L.NT * L.NSG * 16;
  if (e == cudaSuccess) {
    pack_codes_kernel<<<grid_for(nwords, B), B>>>(q, K, N, L.NT, L.UPS, nwords,
                                                  reinterpret_cast<uint32_t*>(p->base + L.codes_off));
    pack_scales_kernel<<<grid_for(npairs, B), B>>>(s, K / g, N, L.NT, npairs,
                                                   reinterpret_cast<uint32_t*>(p->base + L.scales_off));
    pack_zeros_kernel<<<grid_for(nzb, B), B>>>(z, K / g, N, L.NT, nzb, p->base + L.zeros_off);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = pack_error_bits(&bits, true);
  if (e != cudaSuccess) {
    cudaFree(p->base);
    delete p;
    return TM_ERR_CUDA;
  }
  if (bits & kErrBadCode) {
    cudaFree(p->base);
    delete p;
    return TM_ERR_BAD_CODE;
  }
  // Tensor maps for the prefill kernel, one box = one 64-k unit (or its
  // group's scales / the pair's zeros) of 16 consecutive n-tiles:
  //   codes  u32 {128, UPS, NT, NSG}   box {128, 1, 16, 1}
  //   scales u16 {16, 2, NT, NSG}      box {16, 1, 16, 1}
  //   zeros  u8  {16, NT, NSG}         box {16, 16, 1}
  const uint64_t cd[4] = {128, (uint64_t)L.UPS, (uint64_t)L.NT, (uint64_t)L.NSG};
  const uint64_t cs[3] = {kUnitBytes, (uint64_t)L.UPS * kUnitBytes, (uint64_t)L.NT * L.UPS * kUnitBytes};
  const uint32_t cb[4] = {128, 1, 16, 1};
  const uint64_t sd[4] = {16, 2, (uint64_t)L.NT, (uint64_t)L.NSG};
  const uint64_t ss[3] = {32, 64, (uint64_t)L.NT * 64};
  const uint32_t sb[4] = {16, 1, 16, 1};
  const uint64_t zd[3] = {16, (uint64_t)L.NT, (uint64_t)L.NSG};
  const uint64_t zs[2] = {16, (uint64_t)L.NT * 16};
  const uint32_t zb[3] = {16, 16, 1};
  // Tensor-memory kernel, 8 n-tiles a box; a unit is viewed as 4 rows of
  // 128 bytes (8 lanes each) so that the 128-byte swizzle applies:
  //   codes  u32 {32, 4, UPS, NT, NSG} box {32, 4, 1, 8, 1}, 128-byte swizzle
  //   scales u16 {16, 2, NT, NSG}      box {16, 1, 8, 1}
  //   zeros  u8  {16, NT, NSG}         box {16, 8, 1}
  const uint64_t td[5] = {32, 4, (uint64_t)L.UPS, (uint64_t)L.NT, (uint64_t)L.NSG};
  const uint64_t ts[4] = {128, kUnitBytes, (uint64_t)L.UPS * kUnitBytes, (uint64_t)L.NT * L.UPS * kUnitBytes};
  const uint32_t tb[5] = {32, 4, 1, 8, 1};
  const uint32_t tsb[4] = {16, 1, 8, 1};
  const uint32_t tzb[3] = {16, 8, 1};
  bool ok = encode_nd(&p->tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, p->base + L.codes_off, 4, cd, cs, cb) &&
            encode_nd(&p->tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, p->base + L.scales_off, 4, sd, ss, sb) &&
            encode_nd(&p->tm_zeros, CU_TENSOR_MAP_DATA_TYPE_UINT8, p->base + L.zeros_off, 3, zd, zs, zb) &&
            encode_nd(&p->tc_codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, p->base + L.codes_off, 5, td, ts, tb,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_nd(&p->tc_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, p->base + L.scales_off, 4, sd, ss, tsb) &&
            encode_nd(&p->tc_zeros, CU_TENSOR_MAP_DATA_TYPE_UINT8, p->base + L.zeros_off, 3, zd, zs, tzb);
  if (!ok) {
    cudaFree(p->base);
    delete p;
    return TM_ERR_CUDA;
  }
  *out = p;
  return TM_OK;
}

extern "C" tm_status tm_unpack_weights(const tm_packed* p, uint8_t* q, uint8_t* z, uint16_t* s) {
  if (!p || !q || !z || !s) return TM_ERR_INVALID_ARG;
  const Layout& L = p->L;
  const int B = 256;
  const long long nq = (long long)L.K * L.N;
  const long long nm = (long long)(L.K / L.g) * L.N;
  unpack_codes_kernel<<<grid_for(nq, B), B>>>(reinterpret_cast<const uint32_t*>(p->base + L.codes_off), L.K, L.N,
                                              L.NT, L.UPS, q);
  unpack_meta_kernel<<<grid_for(nm, B), B>>>(reinterpret_cast<const uint16_t*>(p->base + L.scales_off),
                                             p->base + L.zeros_off, L.K / L.g, L.N, L.NT, z, s);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

extern "C" tm_status tm_packed_info(const tm_packed* p, int* K, int* N, int* g, size_t* bytes) {
  if (!p) return TM_ERR_INVALID_ARG;
  if (K) *K = p->L.K;
  if (N) *N = p->L.N;
  if (g) *g = p->L.g;
  if (bytes) *bytes = p->L.total;
  return TM_OK;
}

extern "C" void tm_packed_free(tm_packed* p) {
  if (!p) return;
  cudaFree(p->base);
  delete p;
}
