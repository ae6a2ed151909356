// noalloc.cu -- a batch-1 sparse decode entry point that allocates nothing.
//
// Who needs it: code that must not call cudaMalloc while it runs. Examples
// are an inference server that hands out all device memory up front from
// its own pool, code inside a CUDA stream capture (allocation is not allowed
// there), and callers running under a hard memory cap where a surprise
// allocation would fail late. si_sparse_ffn_decode keeps its scratch in the
// layer handle and allocates the library's device error word on first use;
// this entry point keeps both in a fixed array in device memory instead.
//
// The scratch is the 64-bit fixed-point accumulator of the output row (one
// word per output element), the ticket that elects the CTA which converts it
// to float, and two error words: one the launch's bounded waits watch, one
// that si_device_error() reports. The kernel is the same batch-1 decode kernel
// si_sparse_ffn_decode uses; only the scratch pointers differ.
#include <mutex>
#include <string>

#include "../../include/si.h"
#include "common.cuh"
#include "internal.h"

namespace {

// Largest output width this entry point accepts.
constexpr int kNoAllocMaxD = 4096;

// [0, kNoAllocMaxD): accumulator words; word kNoAllocMaxD: the ticket (low
// half); word kNoAllocMaxD + 1: the reported error word (low half) and the
// launch's own error word (high half). Every GPU that loads the library holds
// these 32 KB until the process exits. The accumulator, the ticket and the
// launch's error word must be zero when a call starts: they are zero at load,
// and every call's last CTA sets them back to zero, moving any failure the
// launch recorded (a position outside the packed records, a wait that ran out,
// a partial beyond the accumulator's range) into the reported word first. The
// kernel's bounded waits watch only the launch's own word, so one failed call
// does not cut short the waits of the calls after it. si_device_error() reads
// the reported word (together with the library's other error word) and, on
// request, clears it.
static __device__ __align__(256) unsigned long long g_noalloc_scratch[kNoAllocMaxD + 2];

std::mutex g_noalloc_mu;
unsigned long long* g_noalloc_ptr[128] = {};  // device address of the array, per device

int fail(int code, const char* msg) {
    si::set_error_message(msg);
    return code;
}

// The array's name is only a host-side stand-in; the kernel needs its device
// address, looked up once per device with that device current.
int scratch_for_current_device(unsigned long long** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SI_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= 128) return fail(SI_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return fail(SI_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
        g_noalloc_ptr[dev] = static_cast<unsigned long long*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return SI_OK;
}

}  // namespace

namespace si {
int noalloc_error_word(unsigned** out) {
    unsigned long long* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    *out = reinterpret_cast<unsigned*>(scratch + kNoAllocMaxD + 1);
    return SI_OK;
}
}  // namespace si

extern "C" int si_sparse_ffn_decode_noalloc(const uint16_t* packed, int n_records, int d, const int32_t* S,
                                            int n_sel, const uint16_t* x, float* y, void* stream) {
    if (!packed || (!S && n_sel > 0) || !x || !y) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (n_records < 1 || n_sel < 0) return fail(SI_ERR_INVALID_ARG, "need n_records >= 1 and n_sel >= 0");
    if (d < 256 || d % 64) return fail(SI_ERR_INVALID_ARG, "need d >= 256 and d % 64 == 0");
    if (d > kNoAllocMaxD) return fail(SI_ERR_INVALID_ARG, "d exceeds the no-allocation scratch (4096)");
    const int R = si::sparse_decode_b1_stages(d);
    if (R < 8) return fail(SI_ERR_UNSUPPORTED, "d does not fit the batch-1 decode ring");
    unsigned long long* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    si::SparseDecodeParams P = {};
    P.packed = packed;
    P.n_records = n_records;
    P.d = d;
    P.pos = S;
    P.pmask = nullptr;
    P.n_dev = nullptr;
    P.n_host = n_sel;
    P.x = x;
    P.y = y;
    P.part = nullptr;
    P.part_floats = 0;
    P.tickets = nullptr;
    P.acc = scratch;
    P.acc_ticket = reinterpret_cast<unsigned*>(scratch + kNoAllocMaxD);
    P.err = reinterpret_cast<unsigned*>(scratch + kNoAllocMaxD + 1) + 1;       // this launch's failures
    P.err_report = reinterpret_cast<unsigned*>(scratch + kNoAllocMaxD + 1);   // what si_device_error reads
    P.R = R;
    P.stable_plan = 0;
    P.accumulate = 0;
    const cudaError_t e = si::launch_sparse_decode(P, 1, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        si::set_error_message((std::string("launch failed: ") + cudaGetErrorString(e)).c_str());
        return SI_ERR_CUDA;
    }
    return SI_OK;
}
