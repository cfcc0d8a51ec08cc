// Pieces shared by the tcgen05 kernels (forward and backward): instruction
// and shared-memory descriptors, the bounded mbarrier waiter, and 16-bit
// packing of fp32 pairs.
#pragma once
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
using namespace ptx;

// Instruction descriptor for tcgen05.mma .kind::f16 (PTX ISA, "Instruction
// descriptor"): fp32 accumulator, A/B fp16 or bf16, A K-major, B K- or MN-major.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int M, int N, bool b_mn_major) {
    return (1u << 4)                                  // D format: f32
           | ((bf16 ? 1u : 0u) << 7)                  // A format
           | ((bf16 ? 1u : 0u) << 10)                 // B format
           | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
           | ((uint32_t)(N >> 3) << 17)               // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Shared-memory matrix descriptor (PTX ISA, "Shared memory descriptor"):
// 128-byte swizzle, byte offsets given unencoded.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // SWIZZLE_128B
    return d;
}

struct Waiter {
    volatile int* abort;
    int* status;
    unsigned long long limit;

    // Bounded wait on one phase.  False on timeout (recorded) or if another
    // role already aborted.
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait_nohint(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait_nohint(bar, parity)) return true;
            if ((it & 15u) == 0) {
                if (*abort) return false;
                if (globaltimer_ns() - t0 > limit) {
                    *abort = 1;
                    atomicExch(status, DEV_TIMEOUT);
                    return false;
                }
            }
        }
    }
    // Warp-uniform variant: every lane waits, all lanes agree on the result.
    __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) const {
        bool ok = wait(bar, parity);
        return __all_sync(0xffffffffu, ok);
    }
    // Wait that ignores the abort flag: lets in-flight async work (TMA copies,
    // tcgen05.mma) land before the CTA frees TMEM and its shared memory.  Its
    // bound is kDrainLimitNs whatever the caller set as the ordinary wait
    // limit: work already issued finishes in microseconds, so only a broken
    // device reaches it, and a short ordinary limit can no longer cut a drain
    // short while copies or MMAs are still writing.
    static constexpr unsigned long long kDrainLimitNs = 1000000000ull;  // 1 s
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = globaltimer_ns();
        const unsigned long long bound = limit > kDrainLimitNs ? limit : kDrainLimitNs;
        while (!mbar_try_wait(bar, parity)) {
            if (globaltimer_ns() - t0 > bound) {
                atomicExch(status, DEV_TIMEOUT);
                return;
            }
        }
    }
};

// Bounded waits for a CTA pair: a timeout also raises the other CTA's abort
// flag (written through its shared-memory window) so both halves of the pair
// stop promptly.
struct PairWaiter {
    volatile int* abort;       // this CTA's flag
    volatile int* peer_abort;  // the other CTA's flag
    int* status;
    unsigned long long limit;

    __device__ __forceinline__ void raise() const {
        *abort = 1;
        *peer_abort = 1;
        atomicExch(status, DEV_TIMEOUT);
    }
    // kCluster: acquire at cluster scope, for barriers that take arrivals
    // from threads of the other CTA; barriers signalled by this CTA's threads,
    // by tcgen05.commit or by TMA completion need only CTA scope.
    template <bool kCluster = false>
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        auto probe = [&] { return kCluster ? mbar_try_wait_cl(bar, parity) : mbar_try_wait_nohint(bar, parity); };
        if (probe()) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            if (probe()) return true;
            if ((it & 15u) == 0) {
                if (*abort) return false;
                if (globaltimer_ns() - t0 > limit) {
                    raise();
                    return false;
                }
            }
        }
    }
    template <bool kCluster = false>
    __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) const {
        bool ok = wait<kCluster>(bar, parity);
        return __all_sync(0xffffffffu, ok);
    }
    // Exit-time wait for issued asynchronous work, ignoring the abort flag,
    // bounded by Waiter::kDrainLimitNs from `t0` (one deadline for a whole
    // sequence of drains) or the ordinary limit if that is longer.
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity, uint64_t t0) const {
        const unsigned long long bound = limit > Waiter::kDrainLimitNs ? limit : Waiter::kDrainLimitNs;
        while (!mbar_try_wait_cl_hint(bar, parity)) {
            if (globaltimer_ns() - t0 > bound) {
                atomicExch(status, DEV_TIMEOUT);
                return;
            }
        }
    }
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kBf16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// The two 16-bit values of a packed word, as fp32.
template <bool kBf16>
__device__ __forceinline__ float lo_half(uint32_t w) {
    if (kBf16) return u2f(w << 16);
    float f;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, a;\n\t}" : "=f"(f) : "r"(w));
    return f;
}
template <bool kBf16>
__device__ __forceinline__ float hi_half(uint32_t w) {
    if (kBf16) return u2f(w & 0xFFFF0000u);
    float f;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, b;\n\t}" : "=f"(f) : "r"(w));
    return f;
}

}  // namespace fa
