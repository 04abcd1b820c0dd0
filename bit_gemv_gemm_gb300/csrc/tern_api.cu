// tern_api.cu -- status strings, device checks, host packer/unpacker/validator.
//
// Storage format: each trit t in {-1, 0, +1} in a 2-bit slot, code q = t + 1,
// sixteen slots per little-endian uint32 ("prism-ml/Ternary-Bonsai-27B-mlx-2bit"
// model card, "Memory requirement": each ternary value is stored in a 2-bit slot,
// 2.125 bits per weight with the FP16 scale of each 128-weight group).
#include <atomic>
#include <mutex>

#include "tern_common.cuh"

namespace tern {

namespace {
std::atomic<int> g_last_launches{0};
std::mutex g_dev_mu;
int g_dev_checked[64] = {0};   // 0 = unknown, 1 = ok, -1 = unsupported
int g_dev_sms[64] = {0};
}  // namespace

void set_launch_count(int n) { g_last_launches.store(n, std::memory_order_relaxed); }

tern_status check_device(int* sm_count) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TERN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return TERN_ERR_ARCH;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev_checked[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TERN_ERR_CUDA;
        g_dev_checked[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_dev_sms[dev] = sms;
    }
    if (g_dev_checked[dev] != 1) return TERN_ERR_ARCH;
    if (sm_count) *sm_count = g_dev_sms[dev];
    return TERN_OK;
}

}  // namespace tern

using namespace tern;

extern "C" {

const char* tern_status_str(tern_status s) {
    switch (s) {
        case TERN_OK: return "ok";
        case TERN_ERR_NULL: return "a required pointer is NULL";
        case TERN_ERR_SHAPE: return "shape out of range or not a required multiple";
        case TERN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case TERN_ERR_WORKSPACE: return "workspace missing or too small";
        case TERN_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case TERN_ERR_ARCH: return "the current device is not sm_103 (GB300)";
        case TERN_ERR_DEVICE: return "a kernel reported a device-side error";
    }
    return "unknown status";
}

size_t tern_packed_bytes(int N, int K) {
    if (N < 0 || K < 0 || K % 128 != 0) return 0;
    return (size_t)N * (size_t)K / 4 + (size_t)N * (size_t)K / 64;
}

int tern_last_launch_count(void) { return g_last_launches.load(std::memory_order_relaxed); }

tern_status tern_wait_selftest(int which, int limit_us, tern_stream_t stream) {
    set_launch_count(0);
    if ((which != TERN_SELFTEST_RANGE_FLAG && which != TERN_SELFTEST_MBARRIER) || limit_us < 1 ||
        limit_us > 1000000)
        return TERN_ERR_SHAPE;
    const tern_status d = check_device(nullptr);
    if (d != TERN_OK) return d;
    const uint64_t ns = 1000ull * (uint64_t)limit_us;
    const cudaError_t e = which == TERN_SELFTEST_RANGE_FLAG ? launch_flag_wait_selftest(ns, stream)
                                                            : launch_mbar_wait_selftest(ns, stream);
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}

tern_status tern_device_error(int* code) {
    if (!code) return TERN_ERR_NULL;
    *code = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return TERN_ERR_CUDA;
    int a = 0, b = 0, c = 0;
    if (read_gemm_device_error(&a) != cudaSuccess) return TERN_ERR_CUDA;
    if (read_gemv_device_error(&b) != cudaSuccess) return TERN_ERR_CUDA;
    if (read_f3_device_error(&c) != cudaSuccess) return TERN_ERR_CUDA;
    *code = a ? a : (b ? b : c);
    return TERN_OK;
}

// ---------------------------------------------------------------------------
// Host packer / unpacker / validator.  Word-at-a-time: a 16-entry slice of a
// row becomes one uint32 through a code table indexed by the trit's byte.
// ---------------------------------------------------------------------------

tern_status tern_pack_host(const int8_t* t, int N, int K, uint32_t* codes, long long* bad_count) {
    if (N < 0 || K < 0 || K % 16 != 0) return TERN_ERR_SHAPE;
    if ((N > 0 && K > 0) && (!t || !codes)) return TERN_ERR_NULL;
    long long bad = 0;
    const size_t words = (size_t)N * (size_t)(K / 16);
    for (size_t w = 0; w < words; ++w) {
        const int8_t* src = t + w * 16;
        uint32_t word = 0;
        for (int i = 15; i >= 0; --i) {
            const uint8_t b = (uint8_t)src[i];
            // -1 (0xFF) -> 0, 0 -> 1, +1 -> 2, anything else -> 3 (invalid)
            uint32_t q = (b == 0xFFu) ? 0u : (b == 0u) ? 1u : (b == 1u) ? 2u : 3u;
            bad += (q == 3u);
            word = (word << 2) | q;
        }
        codes[w] = word;
    }
    if (bad_count) *bad_count = bad;
    return TERN_OK;
}

tern_status tern_unpack_host(const uint32_t* codes, int N, int K, int8_t* t, long long* bad_count) {
    if (N < 0 || K < 0 || K % 16 != 0) return TERN_ERR_SHAPE;
    if ((N > 0 && K > 0) && (!t || !codes)) return TERN_ERR_NULL;
    static const int8_t kTrit[4] = {-1, 0, 1, 0};
    long long bad = 0;
    const size_t words = (size_t)N * (size_t)(K / 16);
    for (size_t w = 0; w < words; ++w) {
        uint32_t word = codes[w];
        for (int i = 0; i < 16; ++i, word >>= 2) {
            const uint32_t q = word & 3u;
            bad += (q == 3u);
            t[w * 16 + i] = kTrit[q];
        }
    }
    if (bad_count) *bad_count = bad;
    return TERN_OK;
}

// The 1-bit sibling: bit k%32 of word k/32 is 1 for +1; anything but +-1 is
// counted and stored as -1.
tern_status tern_bin_pack_host(const int8_t* t, int N, int K, uint32_t* words, long long* bad_count) {
    if (N < 0 || K < 0 || K % 32 != 0) return TERN_ERR_SHAPE;
    if ((N > 0 && K > 0) && (!t || !words)) return TERN_ERR_NULL;
    long long bad = 0;
    const size_t nwords = (size_t)N * (size_t)(K / 32);
    for (size_t w = 0; w < nwords; ++w) {
        const int8_t* src = t + w * 32;
        uint32_t word = 0;
        for (int i = 0; i < 32; ++i) {
            const int v = src[i];
            bad += (v != 1 && v != -1);
            word |= (v == 1 ? 1u : 0u) << i;
        }
        words[w] = word;
    }
    if (bad_count) *bad_count = bad;
    return TERN_OK;
}

tern_status tern_bin_unpack_host(const uint32_t* words, int N, int K, int8_t* t) {
    if (N < 0 || K < 0 || K % 32 != 0) return TERN_ERR_SHAPE;
    if ((N > 0 && K > 0) && (!t || !words)) return TERN_ERR_NULL;
    const size_t nwords = (size_t)N * (size_t)(K / 32);
    for (size_t w = 0; w < nwords; ++w)
        for (int i = 0; i < 32; ++i) t[w * 32 + i] = ((words[w] >> i) & 1u) ? (int8_t)1 : (int8_t)-1;
    return TERN_OK;
}

tern_status tern_scales_from_g64_host(const void* s64, int N, int K, void* s128, long long* mismatch) {
    if (N < 0 || K < 0 || K % 128 != 0) return TERN_ERR_SHAPE;
    if ((N > 0 && K > 0) && (!s64 || !s128)) return TERN_ERR_NULL;
    const uint16_t* in = static_cast<const uint16_t*>(s64);
    uint16_t* out = static_cast<uint16_t*>(s128);
    long long bad = 0;
    const size_t groups = (size_t)N * (size_t)(K / 128);
    for (size_t i = 0; i < groups; ++i) {
        bad += in[2 * i] != in[2 * i + 1];
        out[i] = in[2 * i];
    }
    if (mismatch) *mismatch = bad;
    return TERN_OK;
}

size_t tern_bin_packed_bytes(int N, int K) {
    if (N < 0 || K < 0 || K % 128 != 0) return 0;
    return (size_t)N * (size_t)K / 8 + (size_t)N * (size_t)K / 64;
}

tern_status tern_validate_host(const uint32_t* codes, int N, int K, long long* bad_count) {
    if (N < 0 || K < 0 || K % 16 != 0) return TERN_ERR_SHAPE;
    if ((N > 0 && K > 0) && !codes) return TERN_ERR_NULL;
    if (!bad_count) return TERN_ERR_NULL;
    long long bad = 0;
    const size_t words = (size_t)N * (size_t)(K / 16);
    for (size_t w = 0; w < words; ++w) {
        const uint32_t v = codes[w];
        // a slot is 3 iff both of its bits are set
        const uint32_t both = v & (v >> 1) & 0x55555555u;
        bad += __builtin_popcount(both);
    }
    *bad_count = bad;
    return TERN_OK;
}

}  // extern "C"
