// Sharding and gathering of parameters, and the standalone rank-order
// reduction.
//
// "Gather tensor-parallel sharded parameters on read in a trace", Change:
// a gather concatenates the shards along the shard dim (rows for column-
// parallel and fused weights, columns for row-parallel), passes replicated
// tensors through and cuts a vocab-parallel head to org_vocab_size. Every
// such reassembly (and its inverse, sharding) is a set of 2-D block copies,
// so one kernel runs a batch of them: bit-exact, 16-byte vectors when every
// row of a block is 16-byte aligned, bytes otherwise.
#include "common.cuh"
#include "tp_internal.h"

namespace tpk {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_batch_kernel(const CopyBatch b, int blocks_per_desc) {
    const int di = blockIdx.x / blocks_per_desc;
    const int bi = blockIdx.x - di * blocks_per_desc;
    if (di >= b.n) return;
    const CopyDesc d = b.d[di];
    const bool vec = ((reinterpret_cast<uintptr_t>(d.src) | reinterpret_cast<uintptr_t>(d.dst) |
                       (uintptr_t)d.row_bytes | (uintptr_t)d.src_pitch | (uintptr_t)d.dst_pitch) & 15) == 0;
    if (vec) {
        const int64_t per_row = d.row_bytes / 16;
        const int64_t total = d.rows * per_row;
        for (int64_t i = (int64_t)bi * kCopyThreads + threadIdx.x; i < total;
             i += (int64_t)blocks_per_desc * kCopyThreads) {
            const int64_t row = i / per_row, v = i - row * per_row;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (d.src) val = __ldg(reinterpret_cast<const uint4*>(
                static_cast<const char*>(d.src) + row * d.src_pitch) + v);
            reinterpret_cast<uint4*>(static_cast<char*>(d.dst) + row * d.dst_pitch)[v] = val;
        }
    } else {
        const int64_t total = d.rows * d.row_bytes;
        for (int64_t i = (int64_t)bi * kCopyThreads + threadIdx.x; i < total;
             i += (int64_t)blocks_per_desc * kCopyThreads) {
            const int64_t row = i / d.row_bytes, v = i - row * d.row_bytes;
            unsigned char val = 0;
            if (d.src) val = static_cast<const unsigned char*>(d.src)[row * d.src_pitch + v];
            static_cast<unsigned char*>(d.dst)[row * d.dst_pitch + v] = val;
        }
    }
}

cudaError_t launch_copy_batch(const CopyBatch& b, cudaStream_t s) {
    if (b.n == 0) return cudaSuccess;
    int64_t max_bytes = 0;
    for (int i = 0; i < b.n; ++i) max_bytes = max_bytes > b.d[i].rows * b.d[i].row_bytes ? max_bytes : b.d[i].rows * b.d[i].row_bytes;
    // enough CTAs per block copy to cover ~4 waves of 152 SMs in total
    int64_t per = (max_bytes / 16 + kCopyThreads - 1) / kCopyThreads;
    int64_t cap = (4 * kSMs * 8) / b.n + 1;
    int bpd = (int)(per < 1 ? 1 : (per > cap ? cap : per));
    copy_batch_kernel<<<b.n * bpd, kCopyThreads, 0, s>>>(b, bpd);
    return cudaGetLastError();
}

// out = residual + (((p0 + p1) + p2) + ...) + bias, float32, rank order.
__global__ void reduce_partials_kernel(const float* __restrict__ part, const float* resid,
                                       const float* __restrict__ bias, float* out, int N,
                                       int64_t M, int64_t H) {
    const int64_t total = M * H;
    const int64_t plane = M * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc = part[i];
        for (int r = 1; r < N; ++r) acc += part[(int64_t)r * plane + i];
        float v = resid ? resid[i] + acc : acc;
        if (bias) v += bias[i % H];
        out[i] = v;
    }
}

cudaError_t launch_reduce_partials(const float* partials, const float* resid, const float* bias,
                                   float* out, int N, int64_t M, int64_t H, cudaStream_t s) {
    const int64_t total = M * H;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 8 * kSMs * 4) blocks = 8 * kSMs * 4;
    reduce_partials_kernel<<<(int)blocks, 256, 0, s>>>(partials, resid, bias, out, N, M, H);
    return cudaGetLastError();
}

}  // namespace tpk
