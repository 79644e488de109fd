// GPU self-tests of the device primitives, built as a separate test library
// (libattn_selftest.so): one 128x128x128 tcgen05 MMA per operand layout the
// attention kernels use, and the bounded-wait timeout path. Only the tests
// load this library.
//
// Layout modes (A, B: 128 x 128 bf16 row-major in global memory; C fp32):
//   0  C = A B^T   A K-major (TMA), B K-major (TMA)            -- S = Q K^T
//   1  C = A B     A K-major (TMA), B MN-major (TMA)           -- O += P V, B from smem
//   2  C = A B     A from tensor memory, B MN-major (TMA)      -- O += P V
//   3  C = A^T B   A MN-major (TMA), B MN-major (TMA)          -- dQ = dS K
//   4  C = A B^T   A K-major written by threads (swizzled), B K-major (TMA) -- dK from dS^T
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBox = 16384;

__global__ void __launch_bounds__(128, 1)
selftest_mma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int mode,
                    const __nv_bfloat16* A, float* C, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t a_s = base, b_s = base + 2 * kBox;
    const uint32_t bar_load = base + 4 * kBox, bar_mma = bar_load + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 4 * kBox + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 4 * kBox + 20);
    if (base & 1023u) {
        if (tid == 0) *status = 2;
        return;
    }
    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_mma, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;   // C at columns [0,128), A (mode 2) at [128,192)
    const WaitCtx w{abort_flag, status, 1000000000ull};
    const bool a_by_tma = mode != 2 && mode != 4;
    if (tid == 0) {
        mbar_expect_tx(bar_load, (a_by_tma ? 2 : 1) * 2 * kBox);
        for (int hf = 0; hf < 2; ++hf) {
            if (a_by_tma) tma_load_3d(a_s + hf * kBox, &tmA, bar_load, hf * 64, 0, 0);
            tma_load_3d(b_s + hf * kBox, &tmB, bar_load, hf * 64, 0, 0);
        }
    }
    const int r = tid;   // one row per thread
    if (mode == 2) {     // A row r -> tensor memory lane r, two bf16 per column
        uint32_t rr[32];
        const uint32_t* arow = reinterpret_cast<const uint32_t*>(A + r * 128);
        for (int c = 0; c < 2; ++c) {
            for (int i = 0; i < 32; ++i) rr[i] = arow[c * 32 + i];
            tmem_st32(tmem_at(tmem, warp * 32, 128 + c * 32), rr);
        }
        tmem_st_wait();
    } else if (mode == 4) {   // A row r -> swizzled K-major shared-memory tile
        const uint4* arow = reinterpret_cast<const uint4*>(A + r * 128);
        for (int chunk16 = 0; chunk16 < 16; ++chunk16) {
            const int hf = chunk16 >> 3, chunk = chunk16 & 7;
            uint8_t* dst = smem + hf * kBox + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = arow[chunk16];
        }
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after_sync();
        if (mbar_wait(bar_load, 0, w)) {
            const uint32_t idesc =
                idesc_bf16_f32(128, 128, mode == 3, mode == 1 || mode == 2 || mode == 3);
            for (int k = 0; k < 8; ++k) {
                const uint32_t koff = (k >> 2) * kBox + (k & 3) * 32;   // K-major step
                const uint32_t moff = k * 2048;                         // MN-major step
                const uint64_t bdesc = (mode == 0 || mode == 4) ? sdesc_sw128(b_s + koff, 16, 1024)
                                                                : sdesc_sw128(b_s + moff, kBox, 1024);
                if (mode == 2) {
                    mma_ts(tmem, tmem + 128 + k * 8, bdesc, idesc, k > 0);
                } else {
                    const uint64_t adesc = mode == 3 ? sdesc_sw128(a_s + moff, kBox, 1024)
                                                     : sdesc_sw128(a_s + koff, 16, 1024);
                    mma_ss(tmem, adesc, bdesc, idesc, k > 0);
                }
            }
            tc_commit(bar_mma);
        } else {
            // nothing issued: release the waiters below
            mbar_arrive(bar_mma);
        }
    }
    __syncwarp();
    const bool ok = mbar_wait(bar_mma, 0, w);
    tc_fence_after_sync();
    uint32_t rr[32];
    for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem_at(tmem, warp * 32, c * 32), rr);
        if (ok)
            for (int i = 0; i < 32; ++i) C[r * 128 + c * 32 + i] = __uint_as_float(rr[i]);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

// A bounded wait on a barrier nothing will arrive at: must give up, record a
// timeout in *status and return normally.
__global__ void selftest_timeout_kernel(int* status, unsigned long long budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const WaitCtx w{&abort_flag, status, budget_ns};
    if (threadIdx.x == 0) mbar_wait(b, 0, w);
    __syncthreads();
}

// Both exp2 paths of the softmax on an array of inputs.
__global__ void selftest_exp2_kernel(const float* x, float* y_poly, float* y_mufu, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        y_poly[i] = ex2_poly3(x[i]);
        y_mufu[i] = ex2_mufu(x[i]);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A 128 x 128 bf16 row-major matrix as a [128 rows, 1, 128] tensor with 64-column boxes.
bool map128(CUtensorMap* m, const void* ptr) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, 1, 128};
    cuuint64_t strides[2] = {256, 256};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace attn

using namespace attn;

// Returns 0 on launch success; the kernel status word (0 = clean) is written to *status_dev.
extern "C" int attn_selftest_mma(int mode, const void* A, const void* B, float* C, int* status_dev,
                                 cudaStream_t stream) {
    if (mode < 0 || mode > 4) return -1;
    CUtensorMap ta, tb;
    if (!map128(&ta, A) || !map128(&tb, B)) return -3;
    const int smem = 4 * kBox + 64 + 1024;
    if (cudaFuncSetAttribute(selftest_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return -3;
    selftest_mma_kernel<<<1, 128, smem, stream>>>(ta, tb, mode, static_cast<const __nv_bfloat16*>(A), C, status_dev);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

extern "C" int attn_selftest_wait_timeout(int* status_dev, unsigned long long budget_ns, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status_dev, budget_ns);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

// y_poly = FMA-polynomial exp2(x), y_mufu = hardware exp2(x), n elements (device pointers).
extern "C" int attn_selftest_exp2(const float* x, float* y_poly, float* y_mufu, int n, cudaStream_t stream) {
    if (n <= 0) return 0;
    selftest_exp2_kernel<<<(n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024, 256, 0, stream>>>(x, y_poly, y_mufu, n);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
