// Exhaustive check, over every bf16 g with |g| <= 64, of the packed fast path
// and the certificates the fused SwiGLU kernels use (swiglu_math.cuh):
//   * t = e^-g (own exp on ex2.approx) against fp64, in ulps;
//   * s = rcp.approx(1 + t) against fp64 sigma;
//   * silu: every a certified by silu2_cert equals
//     RN_bf16(RN_f32(g * RN_f32(sigma)));
//   * dg: the fast factor si = s (1 + g t s) against F = sigma (1 + g (1 -
//     sigma)).  The kernels accept PG = RN(dyu si) when both ends of
//     PG -+ dyu W round to the same bf16, W = dg2_width(s, go, 1 + go); that
//     is sound when |si - F| plus the roundings of PG and of the interval end
//     (each at most 2^-24 |si| per unit of dyu) stays below W.  dyu is exact
//     in fp32, so this covers every (dy, u) pair.  The sign of si must be the
//     sign of F (it decides the sign of a zero dg).
// Exit status 2 if a certified result is wrong, a margin is too small or a
// sign is wrong.
#include <cstdio>
#include <cstring>
#include "swiglu_math.cuh"
using namespace mx;
using namespace mx::swiglu_math;
struct Out { unsigned t_err, s_err, a_bad, a_fast, dg_ratio, dg_bad, dg_fast, sign_bad; };
__device__ void amaxf(unsigned* p, float v) { atomicMax(p, __float_as_uint(fmaxf(v, 0.f))); }
__global__ void k(Out* o) {
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= 65536) return;
  const float g = __uint_as_float(b << 16);
  if (!(fabsf(g) <= 64.0f)) return;
  const f2 G = f2_pack(g, g);
  const SigFast2 f = sig_fast2(G);
  float t, s, t1, s1; f2_unpack(f.T, t, t1); f2_unpack(f.S, s, s1);
  const double gd = g, et = exp(-gd);
  int ex; frexp(et, &ex);
  amaxf(&o->t_err, (float)(fabs(t - et) / ldexp(1.0, ex - 24)));
  const double sig = 1.0 / (1.0 + et), oms_e = et / (1.0 + et);
  amaxf(&o->s_err, (float)(fabs(s - sig) / sig * 0x1p23));
  // silu: certified results must equal RN_bf16(RN_f32(g * RN_f32(sigma)))
  uint32_t miss;
  const uint32_t A = silu2_cert(G, f.S, miss);
  if ((miss & 0xFFFFu) == 0) {
    atomicAdd(&o->a_fast, 1u);
    const float q = __fmul_rn(g, __double2float_rn(sig));
    if ((A & 0xFFFFu) != f32_to_bf16_bits(q)) atomicAdd(&o->a_bad, 1u);
  }
  // dg: si = s (1 + g (t s)) against F = sigma (1 + g (1 - sigma))
  const f2 GO = f2_mul(G, f2_mul(f.T, f.S));
  const f2 IN = f2_add(GO, f2_splat(1.0f));
  const f2 SI = f2_mul(f.S, IN);
  const f2 W2 = dg2_width(f.S, GO, IN);
  float si, w, x0, x1;
  f2_unpack(SI, si, x0);
  f2_unpack(W2, w, x1);
  atomicAdd(&o->dg_fast, 1u);
  const double F = sig * (1.0 + gd * oms_e);
  const double need = fabs((double)si - F) + 0x1p-23 * 1.01 * fabs((double)si);
  amaxf(&o->dg_ratio, (float)(need / (double)w));
  if (!(need < (double)w)) atomicAdd(&o->dg_bad, 1u);
  if ((si < 0.0f) != (F < 0.0) || si == 0.0f) atomicAdd(&o->sign_bad, 1u);
}
int main() {
  Out* d; cudaMalloc(&d, sizeof(Out)); cudaMemset(d, 0, sizeof(Out));
  k<<<256, 256>>>(d);
  Out h; cudaError_t e = cudaMemcpy(&h, d, sizeof(Out), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) { printf("cuda error %s\n", cudaGetErrorString(e)); return 1; }
  float te, se, dr; memcpy(&te, &h.t_err, 4); memcpy(&se, &h.s_err, 4); memcpy(&dr, &h.dg_ratio, 4);
  printf("t max ulp %.3f; s max rel err %.3f x 2^-23\n", te, se);
  printf("silu: %u certified, %u wrong\n", h.a_fast, h.a_bad);
  printf("dg: %u g on the fast path, max needed/margin %.3f, %u with needed >= margin, %u sign errors\n",
         h.dg_fast, dr, h.dg_bad, h.sign_bad);
  return (h.a_bad || h.dg_bad || h.sign_bad) ? 2 : 0;
}
