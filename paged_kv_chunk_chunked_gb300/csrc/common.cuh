// Device helpers shared by the libpkv kernels: element conversion, error
// reporting and vector memory access.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Codes a kernel writes into the pool's device error word (first writer wins).
enum DeviceError : int {
    kErrNone = 0,
    kErrWaitTimeout = 1,     // a bounded mbarrier / flag wait expired
    kErrBadPage = 2,         // a block-table or selection entry out of range
    kErrTmemAlloc = 3,       // tensor-memory allocation returned an unusable address
    kErrSlots = 4,           // more pages requested for staging than device slots
};

__device__ __forceinline__ void report_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ __forceinline__ static float load(const float* p) { return *p; }
    __device__ __forceinline__ static void store(float* p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, float x) {
        *p = __float2bfloat16_rn(x);
    }
};

// 16-byte vector of elements: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Widen a 16-byte vector to floats (4 for fp32, 8 for bf16).
template <typename T> __device__ __forceinline__ void widen16(const uint4& u, float* f);
template <> __device__ __forceinline__ void widen16<float>(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <> __device__ __forceinline__ void widen16<__nv_bfloat16>(const uint4& u, float* f) {
    f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
    f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

// Pack two floats into a bf16x2 word (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Number of listed pages in a selection row (ascending, -1 padded), by one
// warp: 32 entries per coalesced load; every lane gets the count.
__device__ __forceinline__ int sel_count_warp(const int32_t* row, int kmax, int lane) {
    int n = 0;
    for (int b = 0; b < kmax; b += 32) {
        const int e = b + lane;
        n += __popc(__ballot_sync(0xffffffffu, e < kmax && row[e] >= 0));
    }
    return n;
}

// Vectorised fp32 reduction into global memory (sm_90+ red.global.add.v4.f32).
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace pkv
