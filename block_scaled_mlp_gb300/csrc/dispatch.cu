// dispatch.cu - token-group padding on the device: routed rows -> the padded
// expert-major layout the grouped GEMMs take (offsets and row maps), and a
// row gather that moves bf16 activations into and out of that layout.
//
// Padding layout (pages "[mxfp8] refactor model converter; use token group
// padding kernels in torchao" and "Add MXFP8 fused-MLP overrides in
// torchtitan", Summary): groups in expert order, each group's rows in
// routed-row order, every group padded to a multiple of 128 with zero rows,
// the tail past the last group zero too.
//
// Three launches, no host synchronization:
//   count  each warp owns a chunk of 1024 routed rows and histograms its
//          expert ids in shared memory -> per-chunk counts [chunks, E]
//   scan   one CTA: per-expert totals, padded sizes, exclusive scan over the
//          experts (offsets), then per (chunk, expert) the first padded row
//          of that chunk's rows of that expert (in place over the counts)
//   place  each warp walks its chunk again, 32 rows at a time in order;
//          __match_any_sync groups the lanes that share an expert, a lane's
//          rank among them plus the running per-expert counter in shared
//          memory is its padded row -> stable (rows keep their order).
#include "common.cuh"
#include "kernels.h"

namespace mx {

namespace {

constexpr int TGP_CHUNK = 1024;  // routed rows per warp chunk
constexpr int TGP_WARPS = 8;

__global__ void __launch_bounds__(TGP_WARPS * 32)
    tgp_count_kernel(const int32_t* __restrict__ expert_of, int64_t R, int32_t E, int32_t* __restrict__ counts,
                     int32_t* err) {
  extern __shared__ int32_t hist[];  // [TGP_WARPS][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* h = hist + warp * E;
  const int64_t n_chunks = (R + TGP_CHUNK - 1) / TGP_CHUNK;
  for (int64_t c = (int64_t)blockIdx.x * TGP_WARPS + warp; c < n_chunks; c += (int64_t)gridDim.x * TGP_WARPS) {
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    const int64_t r0 = c * TGP_CHUNK;
    const int64_t r1 = R < r0 + TGP_CHUNK ? R : r0 + TGP_CHUNK;
    bool bad = false;
    for (int64_t r = r0 + lane; r < r1; r += 32) {
      const int32_t e = expert_of[r];
      if (e >= 0 && e < E) atomicAdd(&h[e], 1);
      else bad = true;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) record_error(err, MX_ERR_BAD_OFFSETS);
    __syncwarp();
    for (int e = lane; e < E; e += 32) counts[c * E + e] = h[e];
    __syncwarp();
  }
}

// One CTA of 1024 threads, thread e = expert e.  status[0] = 1 if the
// padded layout fits in M_cap rows.
__global__ void __launch_bounds__(1024)
    tgp_scan_kernel(int32_t* __restrict__ counts, int64_t n_chunks, int32_t E, int32_t pad, int64_t M_cap,
                    int32_t* __restrict__ offs, int32_t* __restrict__ status, int32_t* err) {
  __shared__ long long s[1024];
  const int e = threadIdx.x;
  long long total = 0;
  if (e < E)
    for (int64_t c = 0; c < n_chunks; ++c) total += counts[c * E + e];
  const long long padded = (total + pad - 1) / pad * pad;
  s[e] = e < E ? padded : 0;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan (Hillis-Steele)
    const long long v = e >= off ? s[e - off] : 0;
    __syncthreads();
    s[e] += v;
    __syncthreads();
  }
  const bool fits = s[E - 1] <= M_cap;
  if (e < E) {
    offs[e] = (int32_t)s[e];
    long long run = s[e] - padded;  // first padded row of group e
    for (int64_t c = 0; c < n_chunks; ++c) {
      const int32_t n = counts[c * E + e];
      counts[c * E + e] = (int32_t)run;
      run += n;
    }
  }
  if (e == 0) {
    status[0] = fits ? 1 : 0;
    if (!fits) record_error(err, MX_ERR_BAD_OFFSETS);
  }
}

__global__ void __launch_bounds__(TGP_WARPS * 32)
    tgp_place_kernel(const int32_t* __restrict__ expert_of, int64_t R, int32_t E, const int32_t* __restrict__ base,
                     const int32_t* __restrict__ status, int32_t* __restrict__ row_dst,
                     int32_t* __restrict__ row_src) {
  extern __shared__ int32_t next[];  // [TGP_WARPS][E]: next padded row of each expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* k = next + warp * E;
  const bool fits = status[0] != 0;
  const int64_t n_chunks = (R + TGP_CHUNK - 1) / TGP_CHUNK;
  for (int64_t c = (int64_t)blockIdx.x * TGP_WARPS + warp; c < n_chunks; c += (int64_t)gridDim.x * TGP_WARPS) {
    for (int e = lane; e < E; e += 32) k[e] = base[c * E + e];
    __syncwarp();
    const int64_t r0 = c * TGP_CHUNK;
    const int64_t r1 = R < r0 + TGP_CHUNK ? R : r0 + TGP_CHUNK;
    for (int64_t rb = r0; rb < r1; rb += 32) {
      const int64_t r = rb + lane;
      const int32_t e = r < r1 ? expert_of[r] : -1;
      const bool ok = fits && e >= 0 && e < E;
      // lanes without a valid expert get a key of their own
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, ok ? e : -1 - lane);
      const int32_t pos = ok ? k[e] + __popc(peers & ((1u << lane) - 1u)) : -1;
      __syncwarp();
      if (ok && lane == __ffs(peers) - 1) k[e] += __popc(peers);
      __syncwarp();
      if (r < r1) {
        row_dst[r] = pos;
        if (ok) row_src[pos] = (int32_t)r;
      }
    }
    __syncwarp();
  }
}

// One warp per output row: 16-byte vectors, zeros for negative sources.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint4* __restrict__ x, int64_t rows_in, int64_t vpr, const int32_t* __restrict__ src,
                       int64_t rows_out, int32_t div, uint4* __restrict__ y, int32_t* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t i = (int64_t)blockIdx.x * 8 + warp; i < rows_out; i += (int64_t)gridDim.x * 8) {
    const int32_t s = src[i];
    int64_t t = s >= 0 ? (int64_t)s / div : -1;
    if (t >= rows_in) {
      if (lane == 0) record_error(err, MX_ERR_BAD_OFFSETS);
      t = -1;
    }
    uint4* dst = y + i * vpr;
    if (t < 0) {
      for (int64_t v = lane; v < vpr; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    } else {
      const uint4* row = x + t * vpr;
#pragma unroll 4
      for (int64_t v = lane; v < vpr; v += 32) dst[v] = __ldg(row + v);
    }
  }
}

}  // namespace

size_t token_group_pad_workspace(int64_t R, int32_t E) {
  const int64_t n_chunks = (R + TGP_CHUNK - 1) / TGP_CHUNK;
  return (size_t)(16 + n_chunks * (int64_t)E * 4);
}

int launch_token_group_pad(const int32_t* expert_of, int64_t R, int32_t E, int32_t pad, int64_t M_cap,
                           int32_t* offs, int32_t* row_dst, int32_t* row_src, void* workspace, int32_t* err,
                           cudaStream_t stream) {
  count_launch(MX_KERNEL_MEMSET);
  cudaError_t e = cudaMemsetAsync(row_src, 0xFF, (size_t)M_cap * 4, stream);  // -1: pad and tail
  if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync");
  if (R == 0) {
    count_launch(MX_KERNEL_MEMSET);
    return cuda_status(cudaMemsetAsync(offs, 0, (size_t)E * 4, stream), "cudaMemsetAsync");
  }
  int32_t* status = reinterpret_cast<int32_t*>(workspace);
  int32_t* counts = status + 4;
  const int64_t n_chunks = (R + TGP_CHUNK - 1) / TGP_CHUNK;
  const int grid = (int)std::min<int64_t>((n_chunks + TGP_WARPS - 1) / TGP_WARPS, (int64_t)num_sms() * 4);
  const size_t smem = (size_t)TGP_WARPS * E * 4;
  count_launch(MX_KERNEL_DISPATCH);
  tgp_count_kernel<<<grid, TGP_WARPS * 32, smem, stream>>>(expert_of, R, E, counts, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e, "tgp_count_kernel launch");
  count_launch(MX_KERNEL_DISPATCH);
  tgp_scan_kernel<<<1, 1024, 0, stream>>>(counts, n_chunks, E, pad, M_cap, offs, status, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e, "tgp_scan_kernel launch");
  count_launch(MX_KERNEL_DISPATCH);
  tgp_place_kernel<<<grid, TGP_WARPS * 32, smem, stream>>>(expert_of, R, E, counts, status, row_dst, row_src);
  return cuda_status(cudaGetLastError(), "tgp_place_kernel launch");
}

int launch_gather_rows(const void* x, int64_t rows_in, int64_t cols, const int32_t* src, int64_t rows_out,
                       int32_t div, void* y, int32_t* err, cudaStream_t stream) {
  if (rows_out == 0) return MX_OK;
  const int64_t vpr = cols / 8;
  const int grid = (int)std::min<int64_t>((rows_out + 7) / 8, (int64_t)num_sms() * 16);
  count_launch(MX_KERNEL_DISPATCH);
  gather_rows_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(x), rows_in, vpr, src, rows_out, div,
                                                reinterpret_cast<uint4*>(y), err);
  return cuda_status(cudaGetLastError(), "gather_rows_kernel launch");
}

}  // namespace mx
