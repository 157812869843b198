// layout.cu - the layout / cast / pack kernels around the recurrence:
//   * weight packing into the unit-interleaved 4-slot order the GEMMs and the
//     persistent kernels read (plain, and transposed through 64x64 shared-memory tiles
//     so both sides stay coalesced);
//   * bias packing and bias-gradient scatter back to the caller's gate order;
//   * sequence copies between seq-major [T,B,F] and batch-first [B,T,F], with
//     fp32 <-> bf16 casts, vectorised by four elements;
//   * placing h0 into the output buffer's boundary slot.
// The SystemDS LibMatrixCuDNN.java page does the same job with separate layout
// kernels for the output, the upstream gradients, dx and dW around the cuDNN
// calls of its LSTM forward and backward operators.
#include <type_traits>

#include "common.cuh"

namespace rnn {

namespace {

// Several layout jobs in one launch: job j takes blocks [start[j], start[j+1])
// and walks its elements with a stride of its block count.
//   PACK_ROWS    out[(4u+s)*ld + k] = W[(map[s]*H + u)*K + k]   (zero for map -1)
//   PACK_ROWS_T  out[k*ld + 4u+s]   = the same, through a 64x65 tile
//   PACK_BIAS    out[4u+s] = b[map[s]*H + u]                     (fp32 out)
//   SCATTER_DB   out[map[s]*H + u] = db[4u+s]                    (fp32)
//   H0_TO_Y      Y[slot][b][dir*H + u] = h0[b][u], slot 0 (forward) / T+1 (reverse)
struct PackBatchArgs {
  int n;
  int start[kMaxPackJobs + 1];
  PackJob job[kMaxPackJobs];
};

template <typename T>
__device__ __forceinline__ void pack_job_rows(const PackJob& J, int blk, int nblk) {
  const T* W = static_cast<const T*>(J.in);
  T* out = static_cast<T*>(J.out);
  // 16-byte vectors when the rows allow it (K and ld_out multiples of the
  // vector, 16-byte aligned bases), else one element at a time
  constexpr int V = 16 / static_cast<int>(sizeof(T));
  const bool vec = J.K % V == 0 && J.ld_out % V == 0 && (reinterpret_cast<uintptr_t>(W) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  const int per_row = vec ? J.K / V : J.K;
  const int64_t total = static_cast<int64_t>(4) * J.H * per_row;
  for (int64_t i = static_cast<int64_t>(blk) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(nblk) * blockDim.x) {
    const int row = static_cast<int>(i / per_row), c = static_cast<int>(i - static_cast<int64_t>(row) * per_row);
    const int u = row >> 2, sb = J.map[row & 3];
    if (vec) {
      const uint4 v = sb >= 0 ? *reinterpret_cast<const uint4*>(W + (static_cast<int64_t>(sb) * J.H + u) * J.K + c * V)
                              : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(out + static_cast<int64_t>(row) * J.ld_out + c * V) = v;
    } else {
      out[static_cast<int64_t>(row) * J.ld_out + c] =
          sb >= 0 ? W[(static_cast<int64_t>(sb) * J.H + u) * J.K + c] : from_f<T>(0.0f);
    }
  }
}

// Transposed packing through 64 x 64 tiles: every global access moves two
// consecutive elements (4 bytes for bf16), on the read side along K, on the
// write side along the packed rows (odd K, odd row stride or unaligned
// bases: one element at a time).
template <typename T>
__device__ __forceinline__ void pack_job_rows_t(const PackJob& J, int blk, int nblk, float (*tile)[65]) {
  const T* W = static_cast<const T*>(J.in);
  T* out = static_cast<T*>(J.out);
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
  const int R = 4 * J.H;
  const int tk = (J.K + 63) / 64, tr = (R + 63) / 64;
  using T2 = typename std::conditional<std::is_same<T, float>::value, float2, __nv_bfloat162>::type;
  const bool pair = J.K % 2 == 0 && J.ld_out % 2 == 0 && (reinterpret_cast<uintptr_t>(W) & 7) == 0 &&
                    (reinterpret_cast<uintptr_t>(out) & 7) == 0;
  for (int tile_i = blk; tile_i < tk * tr; tile_i += nblk) {
    const int k0 = (tile_i % tk) * 64, r0 = (tile_i / tk) * 64;
    __syncthreads();
    // rows r0..r0+63 of the packed order, K columns k0..k0+63: tile[row][k]
    for (int i = ty; i < 64; i += 8) {
      const int row = r0 + i;
      const int sb = row < R ? J.map[row & 3] : -1;
      const T* src = sb >= 0 ? W + (static_cast<int64_t>(sb) * J.H + (row >> 2)) * J.K : nullptr;
      const int k = k0 + 2 * tx;
      float v0 = 0.f, v1 = 0.f;
      if (src) {
        if (pair && k + 1 < J.K) {
          const T2 q = *reinterpret_cast<const T2*>(src + k);
          if constexpr (std::is_same<T, float>::value) { v0 = q.x; v1 = q.y; }
          else { const float2 f = __bfloat1622float2(q); v0 = f.x; v1 = f.y; }
        } else {
          if (k < J.K) v0 = to_f<T>(src[k]);
          if (k + 1 < J.K) v1 = to_f<T>(src[k + 1]);
        }
      }
      tile[i][2 * tx] = v0;
      tile[i][2 * tx + 1] = v1;
    }
    __syncthreads();
    // out[k][r0..r0+63]: two consecutive packed rows per thread
    for (int i = ty; i < 64; i += 8) {
      const int k = k0 + i, row = r0 + 2 * tx;
      if (k >= J.K) continue;
      T* dst = out + static_cast<int64_t>(k) * J.ld_out + row;
      const float v0 = tile[2 * tx][i], v1 = tile[2 * tx + 1][i];
      if (pair && row + 1 < R) {
        if constexpr (std::is_same<T, float>::value) *reinterpret_cast<float2*>(dst) = make_float2(v0, v1);
        else *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(v0, v1);
      } else {
        if (row < R) dst[0] = from_f<T>(v0);
        if (row + 1 < R) dst[1] = from_f<T>(v1);
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) pack_batch_kernel(PackBatchArgs P) {
  __shared__ float tile[64][65];
  int j = 0;
  while (j < P.n - 1 && static_cast<int>(blockIdx.x) >= P.start[j + 1]) ++j;
  const PackJob& J = P.job[j];
  const int blk = blockIdx.x - P.start[j], nblk = P.start[j + 1] - P.start[j];
  const int tid = blk * blockDim.x + threadIdx.x, nthr = nblk * blockDim.x;
  switch (J.kind) {
    case PACK_ROWS: pack_job_rows<T>(J, blk, nblk); break;
    case PACK_ROWS_T: pack_job_rows_t<T>(J, blk, nblk, tile); break;
    case PACK_BIAS:
      for (int i = tid; i < 4 * J.H; i += nthr) {
        const int sb = J.map[i & 3];
        static_cast<float*>(J.out)[i] =
            (sb >= 0 && J.in) ? to_f<T>(static_cast<const T*>(J.in)[static_cast<int64_t>(sb) * J.H + (i >> 2)]) : 0.f;
      }
      break;
    case SCATTER_DB:
      for (int i = tid; i < 4 * J.H; i += nthr) {
        const int d = J.map[i & 3];
        if (d >= 0) static_cast<float*>(J.out)[static_cast<int64_t>(d) * J.H + (i >> 2)] =
            static_cast<const float*>(J.in)[i];
      }
      break;
    default: {   // H0_TO_Y
      const int slot = J.dir == 0 ? 0 : J.T + 1;
      for (int i = tid; i < J.B * J.H; i += nthr) {
        const int b = i / J.H, u = i - b * J.H;
        static_cast<T*>(J.out)[(static_cast<int64_t>(slot) * J.B + b) * J.D * J.H + J.dir * J.H + u] =
            J.in ? static_cast<const T*>(J.in)[i] : from_f<T>(0.0f);
      }
    }
  }
}

// One output row (t, b) per blockIdx.x, features along threads.
// Rows (t, b) with t >= len[b] (len non-null) are written as zeros.
template <typename Ti, typename To, int V>
__global__ void seq_copy_kernel(const Ti* __restrict__ in, To* __restrict__ out, int T, int B, int F,
                                int in_bf, int out_bf, int64_t out_ld, const int* __restrict__ len) {
  const int64_t r = blockIdx.x;             // output row index in output order
  int t, b;
  if (out_bf) { b = static_cast<int>(r / T); t = static_cast<int>(r % T); }
  else { t = static_cast<int>(r / B); b = static_cast<int>(r % B); }
  const int64_t ir = in_bf ? (static_cast<int64_t>(b) * T + t) : (static_cast<int64_t>(t) * B + b);
  const Ti* src = in + ir * F;
  To* dst = out + r * out_ld;
  const bool live = !len || t < len[b];
  for (int f = threadIdx.x * V; f < F; f += blockDim.x * V) {
#pragma unroll
    for (int v = 0; v < V; ++v) dst[f + v] = from_f<To>(live ? to_f<Ti>(src[f + v]) : 0.0f);
  }
}

// Recomputation of the LSTM cell states from the saved gate activations
// (the popnn Lstm.cpp page's recomputation mode: previous cell state times the
// forget gate plus input gate times candidate, before the backward pass): one thread per (direction,
// sequence, unit) walks the direction's time order, c_t = f * clip(c_{t-1}) +
// i * g (clip = identity without cell clipping; a masked step t >= len[b]
// keeps c), and writes every c_t in the layout the forward kernels use,
// C[d][slot][b][u] with slot t + 1 (forward direction) or t (reverse) and the
// initial state in slot 0 / T.  Gate loads of four steps are issued before
// their arithmetic.
template <typename T>
__global__ void recompute_cells_kernel(const T* __restrict__ gates, const T* __restrict__ c0, float* __restrict__ C,
                                       int TT, int B, int H, int D, const int* __restrict__ len, int clip, float lo,
                                       float hi) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(D) * B * H) return;
  const int u = static_cast<int>(i % H);
  const int b = static_cast<int>((i / H) % B);
  const int d = static_cast<int>(i / (static_cast<int64_t>(H) * B));
  const int lenb = len ? len[b] : TT;
  float* Cd = C + static_cast<int64_t>(d) * (TT + 1) * B * H;
  float c = c0 ? to_f<T>(c0[(static_cast<int64_t>(d) * B + b) * H + u]) : 0.f;
  Cd[(static_cast<int64_t>(d ? TT : 0) * B + b) * H + u] = c;
  const T* G = gates + (static_cast<int64_t>(d) * TT * B + b) * 4 * H + 4 * u;
  const int64_t gstep = static_cast<int64_t>(B) * 4 * H;
  for (int s0 = 0; s0 < TT; s0 += 4) {
    float g4[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = s0 + j;
      const int t = d ? TT - 1 - s : s;
      if (s < TT) Vec4<T>::load(G + static_cast<int64_t>(t) * gstep, g4[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = s0 + j;
      if (s >= TT) break;
      const int t = d ? TT - 1 - s : s;
      const float cc = clip ? (c < lo ? lo : (c > hi ? hi : c)) : c;
      if (t < lenb) c = g4[j][1] * cc + g4[j][0] * g4[j][2];
      Cd[(static_cast<int64_t>(d ? t : t + 1) * B + b) * H + u] = c;
    }
  }
}

int check_launch() {
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int launch_seq_transpose(const void* in, void* out, int T, int B, int F, int in_bf16, int out_bf16,
                         int in_batch_first, int out_batch_first, int64_t out_ld, cudaStream_t s, const int* len) {
  const int64_t rows = static_cast<int64_t>(T) * B;
  if (rows == 0 || F == 0) return 0;
  if (rows > 0x7fffffffLL) return 2;
  const int vec = (F % 4 == 0 && out_ld % 4 == 0) ? 4 : 1;
  int threads = (F / vec + 31) / 32 * 32;
  if (threads > 256) threads = 256;
  if (threads < 32) threads = 32;
  dim3 grid(static_cast<unsigned>(rows));
#define RNN_SEQ_COPY(TI, TO)                                                                    \
  do {                                                                                          \
    if (vec == 4)                                                                               \
      seq_copy_kernel<TI, TO, 4><<<grid, threads, 0, s>>>(static_cast<const TI*>(in),           \
          static_cast<TO*>(out), T, B, F, in_batch_first, out_batch_first, out_ld, len);        \
    else                                                                                        \
      seq_copy_kernel<TI, TO, 1><<<grid, threads, 0, s>>>(static_cast<const TI*>(in),           \
          static_cast<TO*>(out), T, B, F, in_batch_first, out_batch_first, out_ld, len);        \
  } while (0)
  if (in_bf16 && out_bf16) RNN_SEQ_COPY(__nv_bfloat16, __nv_bfloat16);
  else if (in_bf16) RNN_SEQ_COPY(__nv_bfloat16, float);
  else if (out_bf16) RNN_SEQ_COPY(float, __nv_bfloat16);
  else RNN_SEQ_COPY(float, float);
#undef RNN_SEQ_COPY
  return check_launch();
}

int launch_recompute_cells(const void* gates, const void* c0, float* C, int T, int B, int H, int D, int is_bf16,
                           const int* len, int clip, float lo, float hi, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(D) * B * H;
  const unsigned grid = static_cast<unsigned>((n + 255) / 256);
  if (is_bf16)
    recompute_cells_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(gates),
                                                               static_cast<const __nv_bfloat16*>(c0), C, T, B, H,
                                                               D, len, clip, lo, hi);
  else
    recompute_cells_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(gates),
                                                       static_cast<const float*>(c0), C, T, B, H, D, len, clip, lo,
                                                       hi);
  return check_launch();
}

int launch_pack_batch(const PackBatch& pb, int is_bf16, cudaStream_t s) {
  if (pb.n <= 0) return 0;
  if (pb.n > kMaxPackJobs) return 2;
  PackBatchArgs P;
  P.n = pb.n;
  P.start[0] = 0;
  for (int j = 0; j < pb.n; ++j) {
    const PackJob& J = pb.job[j];
    P.job[j] = J;
    int64_t work;
    switch (J.kind) {
      case PACK_ROWS: work = (static_cast<int64_t>(4) * J.H * J.K + 1023) / 1024; break;
      case PACK_ROWS_T: work = static_cast<int64_t>((J.K + 63) / 64) * ((4 * J.H + 63) / 64); break;
      case H0_TO_Y: work = (static_cast<int64_t>(J.B) * J.H + 255) / 256; break;
      default: work = (4 * J.H + 255) / 256;
    }
    const int nb = static_cast<int>(work < 1 ? 1 : work > 512 ? 512 : work);
    P.start[j + 1] = P.start[j] + nb;
  }
  if (is_bf16) pack_batch_kernel<__nv_bfloat16><<<P.start[pb.n], 256, 0, s>>>(P);
  else pack_batch_kernel<float><<<P.start[pb.n], 256, 0, s>>>(P);
  return check_launch();
}

int launch_fill_zero(void* p, size_t bytes, cudaStream_t s) {
  if (bytes == 0 || p == nullptr) return 0;
  return cudaMemsetAsync(p, 0, bytes, s) == cudaSuccess ? 0 : 3;
}

}  // namespace rnn
