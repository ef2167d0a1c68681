// Decode attention that allocates nothing: mk_attention_decode_noalloc.
//
// Some callers cannot call cudaMalloc at all once they are running: inference
// servers and plugins that hand every byte of HBM to their own pool at start
// up and forbid device allocations afterwards, and latency-critical loops
// where cudaMalloc / cudaFree may synchronise the device and stall other
// streams.  For them this entry point runs one decode step of the attention
// op (RoPE-append of the new key/value row, split-KV partials, log-sum-exp
// combine -- the same computation mk_add_attention lowers to) with its
// partial (m, l, o) scratch in a fixed, file-scope device array instead of a
// caller- or library-allocated buffer.  It uses no library-owned tables
// either: RoPE angles are evaluated in the kernel, in double precision.
//
// The scratch array, kNoallocScratchFloats floats (4 MiB), is part of the
// library image: every GPU that loads the library holds it until the process
// exits.  All calls share it, so calls whose kernels overlap on the GPU (on
// different streams, or from different threads) race on it.  Every slot a
// call reads is written by the same call first, so nothing needs clearing.
// The array's device address is looked up once per device, on the first
// call with that device current, and kept for the life of the process; a
// cudaDeviceReset after that first call is not supported (the reloaded
// module's array may sit elsewhere).
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "graph.h"
#include "mk.h"

namespace mk {
namespace {

constexpr int kNoallocScratchFloats = MK_NOALLOC_SCRATCH_FLOATS;
constexpr int kMaxBatch = 8;
constexpr int kThreadsNA = 256;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

struct NoallocParams {
  const float* qkv;      // [B, (Hq + 2 Hkv) D]
  uint16_t* kc;          // [B, Hkv, cap, D] bf16
  uint16_t* vc;
  float* out;            // [B, Hq D]
  float* scratch;        // device address of g_noalloc_scratch
  int B, Hq, Hkv, D, G, cap;
  double theta;
  int pos[kMaxBatch];    // position of the new token per sequence
  int P[kMaxBatch];      // chunks per sequence
  int slot0[kMaxBatch];  // first slot of (s, kv head 0)
};

__device__ __forceinline__ float bf16_round_to_float(float x) {
  // round to nearest even at 16 bits, as the cache stores it
  const uint32_t u = __float_as_uint(x);
  const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  return __uint_as_float(r);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ float bf16_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Rotate-half RoPE angle pair for dimension i at position pos.
__device__ __forceinline__ void rope_cs(double theta, int D, int i, int pos, float& c, float& s) {
  const double inv = pow(theta, -2.0 * (double)i / (double)D);
  double sd, cd;
  sincos((double)pos * inv, &sd, &cd);
  c = (float)cd;
  s = (float)sd;
}

// One CTA per (sequence, kv head, chunk).  Keys j of the chunk go to warp
// j mod 8; lanes split the head dimension; each warp keeps an online
// softmax per query head (base 2), the 8 warps merge through shared memory.
__global__ void __launch_bounds__(kThreadsNA) noalloc_partial_kernel(const NoallocParams p) {
  extern __shared__ float sm[];
  const int D = p.D, G = p.G, half = D / 2;
  float* qs = sm;                     // [G][D] rotated, scaled q
  float* kn = qs + G * D;             // [D] new key (rotated, bf16-rounded)
  float* vn = kn + D;                 // [D] new value (bf16-rounded)
  float* mrg = vn + D;                // [8][G][D + 2]
  int slot = blockIdx.x, s = 0;
  while (s + 1 < p.B && slot >= p.slot0[s + 1]) ++s;
  const int rel = slot - p.slot0[s];
  const int g = rel / p.P[s], c = rel % p.P[s];
  const int pos = p.pos[s], L = pos + 1, P = p.P[s];
  const int e = (L + P - 1) / P;
  const int j0 = min(c * e, L), j1 = min(j0 + e, L);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* row = p.qkv + (size_t)s * (p.Hq + 2 * p.Hkv) * D;
  const float scale = 1.4426950408889634f / sqrtf((float)D);
  for (int i = tid; i < G * half; i += kThreadsNA) {
    const int h = i / half, j = i % half;
    const float* q = row + (size_t)(g * G + h) * D;
    float cs, sn;
    rope_cs(p.theta, D, j, pos, cs, sn);
    qs[h * D + j] = (q[j] * cs - q[j + half] * sn) * scale;
    qs[h * D + j + half] = (q[j + half] * cs + q[j] * sn) * scale;
  }
  for (int j = tid; j < half; j += kThreadsNA) {
    const float* k = row + (size_t)p.Hq * D + (size_t)g * D;
    float cs, sn;
    rope_cs(p.theta, D, j, pos, cs, sn);
    kn[j] = bf16_round_to_float(k[j] * cs - k[j + half] * sn);
    kn[j + half] = bf16_round_to_float(k[j + half] * cs + k[j] * sn);
  }
  for (int j = tid; j < D; j += kThreadsNA)
    vn[j] = bf16_round_to_float(row[(size_t)(p.Hq + p.Hkv) * D + (size_t)g * D + j]);
  __syncthreads();
  const size_t base = ((size_t)s * p.Hkv + g) * p.cap;
  if (c == 0) {  // the one CTA of (s, g) that stores the new row
    for (int j = tid; j < D; j += kThreadsNA) {
      p.kc[(base + pos) * D + j] = bf16_bits(kn[j]);
      p.vc[(base + pos) * D + j] = bf16_bits(vn[j]);
    }
  }
  const int DPL = D / 32;
  float m[4], l[4], o[4][4], qr[4][4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      o[h][d] = 0.f;
      qr[h][d] = (h < G && d < DPL) ? qs[h * D + lane * DPL + d] : 0.f;
    }
  }
  for (int j = j0 + warp; j < j1; j += 8) {
    float kf[4], vf[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      if (d < DPL) {
        const int dd = lane * DPL + d;
        if (j == pos) {
          kf[d] = kn[dd];
          vf[d] = vn[dd];
        } else {
          kf[d] = bf16_to_float(p.kc[(base + j) * D + dd]);
          vf[d] = bf16_to_float(p.vc[(base + j) * D + dd]);
        }
      } else {
        kf[d] = vf[d] = 0.f;
      }
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if (h < G) {
        float sc = 0.f;
#pragma unroll
        for (int d = 0; d < 4; ++d) sc = fmaf(qr[h][d], kf[d], sc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
        const float mn = fmaxf(m[h], sc);
        const float a = exp2f(m[h] - mn), pe = exp2f(sc - mn);
        l[h] = l[h] * a + pe;
#pragma unroll
        for (int d = 0; d < 4; ++d) o[h][d] = fmaf(o[h][d], a, pe * vf[d]);
        m[h] = mn;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    if (h < G) {
      float* r = mrg + (warp * 4 + h) * (D + 2);
      if (lane == 0) {
        r[0] = m[h];
        r[1] = l[h];
      }
#pragma unroll
      for (int d = 0; d < 4; ++d)
        if (d < DPL) r[2 + lane * DPL + d] = o[h][d];
    }
  }
  __syncthreads();
  float* dst = p.scratch + (size_t)slot * G * (D + 2);
  for (int i = tid; i < G * D; i += kThreadsNA) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
    for (int w = 0; w < 8; ++w) M = fmaxf(M, mrg[(w * 4 + h) * (D + 2)]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < 8; ++w) {
        const float* r = mrg + (w * 4 + h) * (D + 2);
        const float f = exp2f(r[0] - M);
        Ls = fmaf(r[1], f, Ls);
        O = fmaf(r[2 + d], f, O);
      }
    }
    dst[h * (D + 2) + 2 + d] = O;
    if (d == 0) {
      dst[h * (D + 2)] = M;
      dst[h * (D + 2) + 1] = Ls;
    }
  }
}

// One CTA per (sequence, kv head): log-sum-exp merge of its P partials.
__global__ void __launch_bounds__(kThreadsNA) noalloc_combine_kernel(const NoallocParams p) {
  const int s = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
  const int D = p.D, G = p.G, P = p.P[s];
  const float* scr = p.scratch + (size_t)(p.slot0[s] + g * P) * G * (D + 2);
  for (int i = threadIdx.x; i < G * D; i += kThreadsNA) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
    for (int k = 0; k < P; ++k) M = fmaxf(M, scr[(size_t)k * G * (D + 2) + h * (D + 2)]);
    float Ls = 0.f, O = 0.f;
    for (int k = 0; k < P; ++k) {
      const float* r = scr + (size_t)k * G * (D + 2) + h * (D + 2);
      const float f = exp2f(r[0] - M);
      Ls = fmaf(r[1], f, Ls);
      O = fmaf(r[2 + d], f, O);
    }
    p.out[(size_t)s * p.Hq * D + (size_t)(g * G + h) * D + d] = O / Ls;
  }
}

std::mutex g_symbol_mu;
float* g_symbol_ptr[256] = {};  // device address of the scratch array, per device

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" int mk_attention_decode_noalloc(void* stream_, const float* qkv, void* kcache, void* vcache,
                                           float* out, int B, int Hq, int Hkv, int D, int capacity,
                                           const int32_t* pos, const int32_t* len0, int chunk,
                                           double rope_theta) {
  if (!qkv || !kcache || !vcache || !out || !pos || !len0)
    return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: null argument");
  if (B < 1 || B > kMaxBatch) return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: need 1 <= B <= 8");
  if (D != 64 && D != 128) return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: D must be 64 or 128");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > 4)
    return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: need Hq a multiple of Hkv with Hq/Hkv <= 4");
  if (chunk < 0 || capacity < 2 || !(rope_theta > 0.0))
    return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: bad chunk, capacity or rope_theta");
  NoallocParams p{};
  for (int s = 0; s < B; ++s) {
    if (pos[s] < 0 || pos[s] >= capacity)
      return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: pos out of [0, capacity)");
    if (len0[s] < 0 || len0[s] >= capacity)
      return fail(MK_ERR_ARG, "mk_attention_decode_noalloc: len0 out of [0, capacity)");
    p.pos[s] = pos[s];
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
    return fail(MK_ERR_CUDA, "mk_attention_decode_noalloc: no current device");
  if (chunk == 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(MK_ERR_CUDA, "mk_attention_decode_noalloc: cannot query the SM count");
  std::vector<int32_t> l0(len0, len0 + B);
  const std::vector<int> P = partials_per_sequence(l0, Hkv, chunk, sms > 0 ? sms : 1);
  const int G = Hq / Hkv;
  int64_t slots = 0;
  for (int s = 0; s < B; ++s) {
    p.P[s] = P[s];
    p.slot0[s] = (int)slots;
    slots += (int64_t)P[s] * Hkv;
  }
  if (slots * G * (D + 2) > kNoallocScratchFloats)
    return fail(MK_ERR_LIMIT, "mk_attention_decode_noalloc: " + std::to_string(slots * G * (D + 2)) +
                                  " scratch floats needed, limit " + std::to_string(kNoallocScratchFloats));
  float* scratch = nullptr;
  {
    // First call on this device: look up the device address of the array
    // with this device current (host code cannot use the symbol directly).
    std::lock_guard<std::mutex> lk(g_symbol_mu);
    if (!g_symbol_ptr[dev]) {
      void* a = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
      if (e != cudaSuccess)
        return fail(MK_ERR_CUDA, std::string("mk_attention_decode_noalloc: cudaGetSymbolAddress: ") +
                                     cudaGetErrorString(e));
      g_symbol_ptr[dev] = static_cast<float*>(a);
    }
    scratch = g_symbol_ptr[dev];
  }
  p.qkv = qkv;
  p.kc = static_cast<uint16_t*>(kcache);
  p.vc = static_cast<uint16_t*>(vcache);
  p.out = out;
  p.scratch = scratch;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.G = G; p.cap = capacity;
  p.theta = rope_theta;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const size_t smem = (size_t)(G * D + 2 * D + 8 * 4 * (D + 2)) * sizeof(float);
  // an error left by the caller's earlier work stays the caller's: report it
  // without clearing it, and launch nothing
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess)
    return fail(MK_ERR_CUDA, std::string("mk_attention_decode_noalloc: an earlier CUDA error is pending: ") +
                                 cudaGetErrorString(e));
  noalloc_partial_kernel<<<(unsigned)slots, kThreadsNA, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(MK_ERR_CUDA, std::string("mk_attention_decode_noalloc: partial launch: ") + cudaGetErrorString(e));
  noalloc_combine_kernel<<<(unsigned)(B * Hkv), kThreadsNA, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(MK_ERR_CUDA, std::string("mk_attention_decode_noalloc: combine launch: ") + cudaGetErrorString(e));
  return MK_OK;
}
