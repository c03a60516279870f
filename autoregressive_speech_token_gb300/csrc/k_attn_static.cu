// sd_attend_rows_static: the op-level decode attention of sd_attend_rows,
// with its split-KV scratch held in a fixed device array instead of memory
// allocated per call.
//
// Some callers must not allocate device memory while they run: a host thread
// with a hard latency budget (an audio callback cannot absorb cudaMalloc's
// implicit device-wide synchronisation), or an embedding framework that owns
// every byte of device memory through its own pool and forbids raw cudaMalloc.
// They pass inputs and outputs they already own; the partial results live in
// `g_scratch` below.
#include <cstdio>
#include <mutex>

#include "../../include/sd_ops.h"
#include "sd_internal.cuh"

namespace {

// Scratch capacity in floats (4 MiB).  Every device that loads the library
// holds this array until the process exits.
constexpr size_t kScratchFloats = (size_t)1 << 20;

static __device__ __align__(256) float g_scratch[kScratchFloats];
// Positions are passed as an offset from this constant zero, so the call
// needs no host-to-device copy either.
static __device__ int g_zero = 0;

constexpr int kMaxDevices = 64;
struct DevPtrs {
    bool ready = false;
    float* scratch = nullptr;
    int* zero = nullptr;
};
DevPtrs g_dev[kMaxDevices];
std::mutex g_mu;

int err(int code, const char* m, cudaError_t e = cudaSuccess) {
    char buf[256];
    snprintf(buf, sizeof buf, "sd_attend_rows_static: %s%s%s", m, e != cudaSuccess ? ": " : "",
             e != cudaSuccess ? cudaGetErrorString(e) : "");
    sd::set_last_error(buf);
    return code;
}

// Host-side addresses of the two device symbols on the current device.  The
// names g_scratch / g_zero are host stand-ins, not device addresses: only the
// pointers returned by cudaGetSymbolAddress may be given to a kernel.
int device_ptrs(int dev, DevPtrs* out) {
    if (dev < 0 || dev >= kMaxDevices) return err(SD_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DevPtrs& d = g_dev[dev];
    if (!d.ready) {
        cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.scratch), g_scratch);
        if (e != cudaSuccess) return err(SD_ERR_CUDA, "cudaGetSymbolAddress(scratch)", e);
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.zero), g_zero);
        if (e != cudaSuccess) return err(SD_ERR_CUDA, "cudaGetSymbolAddress(zero)", e);
        d.ready = true;
    }
    *out = d;
    return SD_OK;
}

}  // namespace

extern "C" {

int sd_attend_rows_static(const float* q_dev, const uint16_t* k_dev, const uint16_t* v_dev, int32_t B, int32_t H,
                          int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n, int32_t nsplit, float* out_dev,
                          void* stream) {
    if (!q_dev || !k_dev || !v_dev || !out_dev || B < 1 || H < 1 || Hkv < 1 || H % Hkv || H / Hkv > 4 ||
        (hd != 64 && hd != 128) || n < 1 || n > n_ctx || nsplit < 1 || nsplit > 64)
        return err(SD_ERR_INVALID_ARG, "bad argument");
    // scratch: the partials, then one counter per (row, kv head)
    const size_t part_floats = (size_t)B * H * nsplit * sd::part_stride(hd);
    const size_t need = part_floats + (size_t)B * Hkv;
    if (need > kScratchFloats)
        return err(SD_ERR_INVALID_ARG,
                   "B * H * nsplit * (hd + 4) + B * Hkv exceeds the fixed scratch of 1048576 floats");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return err(SD_ERR_CUDA, "cudaGetDevice", e);
    DevPtrs d;
    int rc = device_ptrs(dev, &d);
    if (rc) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    sd::AttnArgs a;
    a.q = q_dev; a.q_stride = H * hd; a.knew = nullptr; a.vnew = nullptr;
    a.kc = reinterpret_cast<__half*>(const_cast<uint16_t*>(k_dev));
    a.vc = reinterpret_cast<__half*>(const_cast<uint16_t*>(v_dev));
    a.row_heads = Hkv; a.head_off = 0; a.n_head = H; a.n_kv = Hkv; a.hd = hd; a.n_ctx = n_ctx; a.nsplit = nsplit;
    a.pos_ptr = d.zero; a.pos_add = n - 1; a.max_len = n; a.part = d.scratch;
    int* counters = reinterpret_cast<int*>(d.scratch + part_floats);
    a.counters = counters; a.out = out_dev; a.out_stride = H * hd;
    // The partial records are written before they are read within a call; the
    // per-(row, kv head) counters must start at zero, so they are cleared here
    // (a previous call that failed part-way could have left them non-zero).
    e = cudaMemsetAsync(counters, 0, sizeof(int) * (size_t)B * Hkv, st);
    if (e == cudaSuccess) e = sd::launch_attention(a, B, st);
    if (e != cudaSuccess) return err(SD_ERR_CUDA, "launch", e);
    // Stream-ordered: no synchronisation here (sd_attend_rows synchronises).  The
    // kernel may still be running; its errors surface at the caller's next
    // synchronisation of `stream`.
    return SD_OK;
}

}  // extern "C"
