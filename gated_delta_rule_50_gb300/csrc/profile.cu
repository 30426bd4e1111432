// profile.cu -- optional per-kernel device timing (see gdn_profile_enable in gdn.h).
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "gdn.h"
#include "profile.h"

namespace gdn {
namespace {
struct Rec {
    const char *name;
    cudaEvent_t a, b;
};
std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t get_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}
}  // namespace

ProfScope::ProfScope(const char *name, cudaStream_t st) : name_(name), st_(st), a_(nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on) return;
    a_ = get_event();
    if (a_) cudaEventRecord(a_, st_);
}

ProfScope::~ProfScope() {
    if (!a_) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = get_event();
    if (!b) return;
    cudaEventRecord(b, st_);
    g_recs.push_back({name_, a_, b});
}

}  // namespace gdn

using namespace gdn;

extern "C" void gdn_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_on = on != 0;
}

extern "C" int gdn_profile_read(char *names, int name_stride, int *counts, double *ms, int max_entries) {
    std::lock_guard<std::mutex> lk(g_mu);
    std::vector<std::string> keys;
    std::vector<int> cnt;
    std::vector<double> tot;
    int rc = 0;
    for (const Rec &r : g_recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) rc = -1;
        size_t i = 0;
        while (i < keys.size() && keys[i] != r.name) ++i;
        if (i == keys.size()) {
            keys.push_back(r.name);
            cnt.push_back(0);
            tot.push_back(0.0);
        }
        cnt[i] += 1;
        tot[i] += t;
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_recs.clear();
    if (rc) return -1;
    int n = 0;
    for (size_t i = 0; i < keys.size() && n < max_entries; ++i, ++n) {
        if (names && name_stride > 0) {
            std::strncpy(names + (size_t)n * name_stride, keys[i].c_str(), name_stride - 1);
            names[(size_t)n * name_stride + name_stride - 1] = '\0';
        }
        if (counts) counts[n] = cnt[i];
        if (ms) ms[n] = tot[i];
    }
    return n;
}
