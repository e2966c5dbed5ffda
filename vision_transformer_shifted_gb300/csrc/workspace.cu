// Handle-owned device workspaces: grown on demand, freed by the handle, and
// two host-side debugging switches read from the environment whenever a
// workspace is (re)allocated:
//   SWIN_WATTN_FAIL_ALLOC  set (and not "0"): every workspace allocation
//       fails as if the device were out of memory, so that callers can test
//       their handling of SWIN_WATTN_ENOMEM without exhausting a GPU;
//   SWIN_WATTN_DEBUG       set (and not "0"): each workspace gets a guard
//       band of GUARD bytes on both sides, filled with a byte pattern; after
//       each call of the entry points that use the workspace the bands are
//       read back (the call then synchronises its stream), and a changed byte
//       -- a kernel writing outside its buffer -- is reported as
//       SWIN_WATTN_ECORRUPT.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "swin_wattn.h"
#include "common.cuh"

namespace swin {

namespace {

constexpr size_t GUARD = 4096;
constexpr unsigned char PATTERN = 0xA5;

std::mutex g_mutex;
// guarded workspaces: the pointer handed out -> (the allocation, its usable bytes)
std::unordered_map<void *, std::pair<void *, size_t>> g_guarded;

bool env_on(const char *name)
{
    const char *v = std::getenv(name);
    return v && *v && std::strcmp(v, "0") != 0;
}

} // namespace

void ws_free(void **buf, size_t *have)
{
    if (*buf) {
        void *raw = *buf;
        {
            std::lock_guard<std::mutex> lock(g_mutex);
            auto it = g_guarded.find(*buf);
            if (it != g_guarded.end()) {
                raw = it->second.first;
                g_guarded.erase(it);
            }
        }
        cudaFree(raw);
    }
    *buf = nullptr;
    *have = 0;
}

int ws_ensure(void **buf, size_t *have, size_t need)
{
    if (*have >= need && *buf) return SWIN_WATTN_OK;
    ws_free(buf, have);
    if (env_on("SWIN_WATTN_FAIL_ALLOC")) return SWIN_WATTN_ENOMEM;
    const bool guarded = env_on("SWIN_WATTN_DEBUG");
    void *raw = nullptr;
    if (cudaMalloc(&raw, guarded ? need + 2 * GUARD : need) != cudaSuccess) {
        cudaGetLastError();
        return SWIN_WATTN_ENOMEM;
    }
    if (!guarded) {
        *buf = raw;
        *have = need;
        return SWIN_WATTN_OK;
    }
    char *p = (char *)raw;
    if (cudaMemset(p, PATTERN, GUARD) != cudaSuccess || cudaMemset(p + GUARD + need, PATTERN, GUARD) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(raw);
        return SWIN_WATTN_ECUDA;
    }
    *buf = p + GUARD;
    *have = need;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_guarded[*buf] = {raw, need};
    return SWIN_WATTN_OK;
}

int ws_check(const void *buf, cudaStream_t stream)
{
    if (!buf) return SWIN_WATTN_OK;
    void *raw = nullptr;
    size_t bytes = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_guarded.empty()) return SWIN_WATTN_OK;
        auto it = g_guarded.find(const_cast<void *>(buf));
        if (it == g_guarded.end()) return SWIN_WATTN_OK;
        raw = it->second.first;
        bytes = it->second.second;
    }
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SWIN_WATTN_ECUDA;
    std::vector<unsigned char> band(2 * GUARD);
    const char *p = (const char *)raw;
    if (cudaMemcpy(band.data(), p, GUARD, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(band.data() + GUARD, p + GUARD + bytes, GUARD, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SWIN_WATTN_ECUDA;
    for (unsigned char c : band)
        if (c != PATTERN) return SWIN_WATTN_ECORRUPT;
    return SWIN_WATTN_OK;
}

int ws_test_corrupt(const void *buf, int side)
{
    void *raw = nullptr;
    size_t bytes = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = g_guarded.find(const_cast<void *>(buf));
        if (it == g_guarded.end()) return SWIN_WATTN_EINVAL;
        raw = it->second.first;
        bytes = it->second.second;
    }
    char *p = (char *)raw + (side ? GUARD + bytes + GUARD - 1 : 0);
    return cudaMemset(p, 0, 1) == cudaSuccess ? SWIN_WATTN_OK : SWIN_WATTN_ECUDA;
}

} // namespace swin
