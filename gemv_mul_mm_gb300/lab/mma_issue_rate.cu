// mma_issue_rate.cu -- measures how fast back-to-back tcgen05.mma kind::f16
// instructions (M = 128, K = 16, fp32 accumulators in tensor memory) run when
// issued from one CTA, to size the prefill GEMM's tiles and its MMA issue path.
// Not part of libqmm.so.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -I include -I gemv_mul_mm_gb300/csrc -o mma_issue_rate gemv_mul_mm_gb300/lab/mma_issue_rate.cu
//   ./mma_issue_rate
//
// Variants:
//   A operand    in tensor memory (tcgen05.mma [d], [a_tmem], b_desc) or in
//                shared memory (a_desc, 128-byte swizzled K-major);
//   N            128 or 256;
//   descriptors  built for every MMA from the stage address, or built once
//                (the 32-byte K steps are +2 on the descriptor);
//   issuers      one thread, or two threads (two warps) each issuing half of
//                the MMAs into its own accumulator.
// One CTA per SM (shared memory forces it), each issuing 8000 MMAs; printed:
// SM cycles per MMA averaged over the CTAs, on 1 CTA and on every SM. The
// operands are random f16 values. Every wait is bounded; a wait that runs
// out is reported and the tensor memory is freed only after a second bounded
// wait.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "sm100_async.cuh"

using namespace qmm;

namespace {

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFF) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d), "r"(a), "l"(b), "r"(idesc),
                 "r"(acc)
                 : "memory");
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d), "l"(a), "l"(b), "r"(idesc),
                 "r"(acc)
                 : "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// A small random f16 pair: codes in [-7, 7] (A) or values in [-2, 2] (B).
__device__ __forceinline__ uint32_t rand_h2(uint32_t i, bool wide) {
    uint32_t h = i * 2654435761u;
    h ^= h >> 15;
    h *= 2246822519u;
    h ^= h >> 13;
    const float a = wide ? (static_cast<int>(h % 2001u) - 1000) / 500.f : static_cast<float>(static_cast<int>(h % 15u) - 7);
    const float b = wide ? (static_cast<int>((h >> 11) % 2001u) - 1000) / 500.f
                         : static_cast<float>(static_cast<int>((h >> 11) % 15u) - 7);
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

constexpr int kIters = 2000;   // 4 MMAs (K = 64) per iteration
constexpr int kA = 16384, kB = 32768;

struct Cfg {
    int a_in_tmem, n, once, issuers;
};

// out[3b..3b+2] = max over the CTA's issuers of {cycles to completion, cycles issuing, timed out}
__global__ void __launch_bounds__(128, 1) k_rate(Cfg c, unsigned long long* out) {
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
    const uint32_t A = smem_u32(sm), B = A + kA;   // 128 x 64 and up to 256 x 64 f16, 128-byte swizzled
    __shared__ uint64_t bar[2];
    __shared__ uint32_t tslot;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (kA + kB) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(sm)[i] = rand_h2(i, i >= kA / 4);
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tslot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_sync();
    const uint32_t tmem = tslot;
    {   // A operand in tensor memory: columns [0, 32) of every lane, random codes
        uint32_t v[32];
        for (int j = 0; j < 32; ++j) v[j] = rand_h2(threadIdx.x * 32 + j + 77777, false);
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
                tmem + (static_cast<uint32_t>(warp * 32) << 16)),
            "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
            "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
            "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
            "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
            : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    tc_sync();
    const uint32_t idesc = (1u << 4) | ((static_cast<uint32_t>(c.n) >> 3) << 17) | ((128u >> 4) << 24);
    const int me = threadIdx.x == 0 ? 0 : (c.issuers == 2 && threadIdx.x == 32) ? 1 : -1;
    if (me >= 0) {
        const uint32_t d = tmem + 128 + me * c.n;   // accumulator columns (two issuers: N = 128 only)
        const int iters = kIters / c.issuers;
        const long long t0 = clock64();
        if (c.once) {
            // the first K = 64 step starts the accumulator; the loop only accumulates
            const uint64_t b0 = desc_sw128(B), a0 = desc_sw128(A);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (c.a_in_tmem)
                    mma_ts(d, tmem + 8 * kk, b0 + 2 * kk, idesc, kk != 0);
                else
                    mma_ss(d, a0 + 2 * kk, b0 + 2 * kk, idesc, kk != 0);
            }
#pragma unroll 1
            for (int it = 1; it < iters; ++it) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (c.a_in_tmem)
                        mma_ts(d, tmem + 8 * kk, b0 + 2 * kk, idesc, 1);
                    else
                        mma_ss(d, a0 + 2 * kk, b0 + 2 * kk, idesc, 1);
                }
            }
        } else {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (c.a_in_tmem)
                        mma_ts(d, tmem + 8 * kk, desc_sw128(B + 32 * kk), idesc, (it | kk) != 0);
                    else
                        mma_ss(d, desc_sw128(A + 32 * kk), desc_sw128(B + 32 * kk), idesc, (it | kk) != 0);
                }
            }
        }
        commit(&bar[me]);
        const long long t1 = clock64();
        unsigned long long to = 0;
        while (!mbar_try_wait(&bar[me], 0)) {
            if (clock64() - t0 > (1ll << 31)) {
                to = 1;
                break;
            }
        }
        const long long t2 = clock64();
        atomicMax(&out[3 * blockIdx.x + 0], static_cast<unsigned long long>(t2 - t0));
        atomicMax(&out[3 * blockIdx.x + 1], static_cast<unsigned long long>(t1 - t0));
        atomicMax(&out[3 * blockIdx.x + 2], to);
        if (to) {   // a second bounded chance for the MMAs before the tensor memory is freed
            const long long t3 = clock64();
            while (!mbar_try_wait(&bar[me], 0) && clock64() - t3 < (1ll << 31)) {
            }
        }
    }
    tc_sync();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

}  // namespace

int main() {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms <= 0) {
        printf("no device\n");
        return 1;
    }
    unsigned long long* d = nullptr;
    cudaMalloc(&d, sizeof(unsigned long long) * 3 * sms);
    const int smem = 160 * 1024;   // more than half an SM's shared memory: one CTA per SM
    cudaFuncSetAttribute(k_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    unsigned long long* h = new unsigned long long[3 * sms];
    printf("%-14s %4s %-9s %-8s %5s %14s %6s\n", "A operand", "N", "desc", "issuers", "CTAs", "cycles/MMA", "ideal");
    for (int a_in_tmem = 1; a_in_tmem >= 0; --a_in_tmem)
        for (int n : {128, 256})
            for (int once = 0; once < 2; ++once)
                for (int issuers = 1; issuers <= 2; ++issuers) {
                    if (issuers == 2 && n == 256) continue;   // two 256-column accumulators do not fit beside A
                    for (int grid : {1, sms}) {
                        const Cfg c = {a_in_tmem, n, once, issuers};
                        cudaMemset(d, 0, sizeof(unsigned long long) * 3 * sms);
                        k_rate<<<grid, 128, smem>>>(c, d);
                        if (cudaDeviceSynchronize() != cudaSuccess) {
                            printf("launch failed: %s\n", cudaGetErrorString(cudaGetLastError()));
                            return 1;
                        }
                        cudaMemcpy(h, d, sizeof(unsigned long long) * 3 * grid, cudaMemcpyDeviceToHost);
                        double tot = 0;
                        unsigned long long timeouts = 0;
                        for (int b = 0; b < grid; ++b) {
                            tot += static_cast<double>(h[3 * b]);
                            timeouts += h[3 * b + 2];
                        }
                        printf("%-14s %4d %-9s %-8d %5d %14.1f %6d%s\n", a_in_tmem ? "tensor memory" : "shared memory", n,
                               once ? "once" : "per MMA", issuers, grid, tot / grid / (4.0 * kIters), n / 2,
                               timeouts ? "  (a wait ran out)" : "");
                    }
                }
    delete[] h;
    cudaFree(d);
    return 0;
}
