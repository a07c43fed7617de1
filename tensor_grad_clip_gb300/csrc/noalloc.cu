// soma_clip_norm_noalloc: the global gradient norm and clip coefficient
// without any memory allocation by the library.
//
// Some callers cannot allocate device memory: a host application or
// framework that owns the whole device heap through its own allocator (a
// stray cudaMalloc there fails once that allocator has reserved HBM, or
// fragments its pool), and latency-critical loops in which cudaMalloc /
// cudaFree, which may synchronise the device, are not allowed.  For them this
// entry point runs the square-sum kernel with all of its scratch (the
// arrival ticket and result, the per-chunk partial sums and the chunk /
// segment tables) placed in one file-scope __device__ array of fixed size.
// The runtime loads this file's device image lazily: the array takes its
// device memory on the first call on a device (when cudaGetSymbolAddress
// loads the image) and keeps it until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (in host code the array's
// name is only a host-side stand-in, not a device address) and caches it.
// Make that first call before any stream capture.
//
// The tables reach the array inside the arguments of small copy kernels:
// a launch copies its arguments when it is enqueued, so the host staging
// buffer is free again as soon as the launches are enqueued, and a call
// returns without waiting for anything on the GPU.
//
// All calls share the one array, which keeps the contents of the last call:
// every call rewrites the tables and clears the result/ticket block before
// launching.  Calls whose work overlaps on the GPU (different streams with no
// ordering between them, or several threads) race on the array; order them.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "soma_kernels.h"
#include "soma_opt.h"

namespace {

constexpr size_t kScratchBytes = SOMA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
constexpr size_t kResultBytes = 256;         // soma::Result, padded
constexpr int64_t kMinChunk = 32768;          // elements per chunk, at least
constexpr int64_t kTargetChunks = 32768;      // grows the chunk for large lists
// 16-byte words of the staged image one copy launch carries in its
// arguments (30,400 bytes; kernel arguments may take up to 32,764).
constexpr int kArgWords = 1900;

// Arguments of one copy launch: `nwords` words for `dst` (16-byte aligned).
struct StageArgs {
    uint4* dst;
    int32_t nwords;
    int32_t pad;
    uint4 words[kArgWords];
};
static_assert(sizeof(StageArgs) <= 32764, "kernel arguments are limited to 32,764 bytes");

__global__ void write_stage_kernel(const __grid_constant__ StageArgs a) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.nwords; i += gridDim.x * blockDim.x)
        a.dst[i] = a.words[i];
}

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_mu;                               // one host-side user at a time
alignas(256) unsigned char g_stage[kScratchBytes];  // host image of the scratch
StageArgs g_args;                              // arguments of the copy launch being enqueued
void* g_dev_scratch[kMaxDevices];              // per device: address of the array

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Counts (segs == nullptr) or writes the norm table: the
// trainable, owned entries cut into segments by the step's own cutting rule
// (soma::segment_cut), grouped into chunks of about `chunk` elements and at
// most kMaxSegsPerChunk segments each.  The vector head is the number of
// leading elements before the gradient is 16-byte aligned.  The step's
// table builder keeps its segments in a growing array; this one writes into
// the fixed staging buffer and allocates nothing.
void norm_table(const soma_tensor_t* list, int64_t n, int64_t chunk, soma::Seg* segs, int32_t* begin,
                int64_t* nseg_out, int64_t* nchunk_out) {
    int64_t nseg = 0, nchunk = 0, cur_elems = 0;
    int cur_segs = 0;
    if (begin) begin[0] = 0;
    for (int64_t k = 0; k < n; ++k) {
        const soma_tensor_t& t = list[k];
        if (!t.trainable || !t.owned || t.numel == 0) continue;
        const int gsz = t.grad_dtype == SOMA_DTYPE_F32 ? 4 : 2;  // fp32, or bf16 / fp16
        int h = -1;
        for (int c = 0; c < soma::kVec && h < 0; ++c)
            if (((uintptr_t)t.grad + (uintptr_t)c * gsz) % 16 == 0) h = c;
        int64_t off = 0;
        while (off < t.numel) {
            if (cur_segs == soma::kMaxSegsPerChunk || cur_elems >= chunk) {
                ++nchunk;
                if (begin) begin[nchunk] = (int32_t)nseg;
                cur_elems = 0;
                cur_segs = 0;
            }
            const int64_t cut = soma::segment_cut(off, t.numel, chunk - cur_elems, h);
            const int64_t len = cut - off;
            if (segs) {
                soma::Seg s{};
                s.g = static_cast<const char*>(t.grad) + off * gsz;
                soma::segment_body(off, len, h, s);
                s.gdtype = t.grad_dtype;
                segs[nseg] = s;
            }
            ++nseg;
            cur_elems += len;
            ++cur_segs;
            off = cut;
        }
    }
    if (cur_segs > 0) {
        ++nchunk;
        if (begin) begin[nchunk] = (int32_t)nseg;
    }
    *nseg_out = nseg;
    *nchunk_out = nchunk;
}

struct CurrentDevice {
    int prev = -1;
    cudaError_t status = cudaSuccess;
    explicit CurrentDevice(int dev) {
        status = cudaGetDevice(&prev);
        if (status == cudaSuccess && prev != dev) status = cudaSetDevice(dev);
    }
    ~CurrentDevice() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" soma_status_t soma_clip_norm_noalloc(int32_t device, const soma_tensor_t* list, int64_t n,
                                                double grad_divisor, double max_norm, double* out,
                                                void* stream) {
    if (device < 0 || device >= kMaxDevices || n < 0 || (n > 0 && !list) || !out ||
        (uintptr_t)out % alignof(double) != 0)
        return SOMA_ERR_INVALID_ARG;
    if (!std::isfinite(grad_divisor) || grad_divisor <= 0 || !std::isfinite(max_norm) || max_norm <= 0)
        return SOMA_ERR_INVALID_ARG;
    int64_t owned = 0;
    for (int64_t k = 0; k < n; ++k) {
        const soma_tensor_t& t = list[k];
        if (t.trainable > 1 || t.owned > 1 || t.numel < 0) return SOMA_ERR_INVALID_ARG;
        if (!t.trainable || !t.owned || t.numel == 0) continue;
        if (t.grad_dtype != SOMA_DTYPE_F32 && t.grad_dtype != SOMA_DTYPE_BF16 && t.grad_dtype != SOMA_DTYPE_F16)
            return SOMA_ERR_DTYPE;
        if (!t.grad) return SOMA_ERR_INVALID_ARG;
        if ((uintptr_t)t.grad % (t.grad_dtype == SOMA_DTYPE_F32 ? 4 : 2)) return SOMA_ERR_ALIGNMENT;
        owned += t.numel;
    }
    int64_t chunk = std::max<int64_t>(kMinChunk, (owned + kTargetChunks - 1) / kTargetChunks);
    chunk = (chunk + 63) / 64 * 64;

    std::lock_guard<std::mutex> lock(g_mu);
    int64_t nseg = 0, nchunk = 0;
    norm_table(list, n, chunk, nullptr, nullptr, &nseg, &nchunk);
    const size_t o_part = kResultBytes;
    const size_t o_seg = o_part + up256((size_t)std::max<int64_t>(nchunk, 1) * sizeof(double));
    const size_t o_beg = o_seg + up256((size_t)nseg * sizeof(soma::Seg));
    const size_t bytes = o_beg + up256((size_t)(nchunk + 1) * sizeof(int32_t));
    if (bytes > kScratchBytes) return SOMA_ERR_LIMIT;  // list needs more scratch than the array holds

    CurrentDevice cd(device);
    if (cd.status != cudaSuccess) return SOMA_ERR_CUDA;
    if (!g_dev_scratch[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SOMA_ERR_CUDA;
        }
        g_dev_scratch[device] = p;
    }
    unsigned char* d = static_cast<unsigned char*>(g_dev_scratch[device]);

    std::memset(g_stage, 0, kResultBytes);  // result and arrival ticket start at zero
    norm_table(list, n, chunk, reinterpret_cast<soma::Seg*>(g_stage + o_seg),
               reinterpret_cast<int32_t*>(g_stage + o_beg), &nseg, &nchunk);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The result block (cleared) and the tables go to the array in the
    // arguments of copy launches, whose arguments are copied at enqueue time:
    // g_stage may be rewritten by the next call as soon as this one returns.
    // The partial sums need no copy; the square-sum kernel writes them.
    const size_t regions[2][2] = {{0, kResultBytes}, {o_seg, bytes}};
    for (const auto& rg : regions) {
        for (size_t off = rg[0]; off < rg[1]; off += sizeof(g_args.words)) {
            const size_t n16 = (std::min(rg[1] - off, sizeof(g_args.words)) + 15) / 16;
            g_args.dst = reinterpret_cast<uint4*>(d + off);
            g_args.nwords = (int32_t)n16;
            std::memcpy(g_args.words, g_stage + off, n16 * 16);
            write_stage_kernel<<<(int)std::min<size_t>(8, (n16 + 255) / 256), 256, 0, s>>>(g_args);
            if (cudaGetLastError() != cudaSuccess) return SOMA_ERR_CUDA;
        }
    }
    soma::NormArgs a{};
    a.t = soma::Table{reinterpret_cast<const soma::Seg*>(d + o_seg), reinterpret_cast<const int32_t*>(d + o_beg),
                      (int32_t)nchunk};
    a.partials = reinterpret_cast<double*>(d + o_part);
    a.res = reinterpret_cast<soma::Result*>(d);
    a.divisor = grad_divisor;
    a.inv_step_divisor = 1.0 / grad_divisor;
    a.max_norm = max_norm;
    for (double& w : a.inv_divisor) w = 1.0 / grad_divisor;  // every segment is group 0 here
    if (soma::launch_norm(a, (int)std::max<int64_t>(nchunk, 1), stream) != cudaSuccess) return SOMA_ERR_CUDA;
    // norm and coef are adjacent in the result block
    if (cudaMemcpyAsync(out, d + offsetof(soma::Result, norm), 2 * sizeof(double), cudaMemcpyDefault, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return SOMA_ERR_CUDA;
    }
    return SOMA_OK;
}
