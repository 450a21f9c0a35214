// Optional per-kernel timing of libmoe launches: when enabled, every kernel
// launch is bracketed by a pair of CUDA events recorded on its own stream, and
// moe_timing_report() turns the pairs into per-kernel counts and milliseconds
// after the caller has synchronised. Disabled (the default) it costs one
// branch per launch.
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "timing.h"

namespace moe {

namespace {
struct Pair {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_mu;
bool g_on = false;
std::vector<Pair> g_pairs;
std::vector<cudaEvent_t> g_free;

cudaEvent_t get_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

LaunchTimer::LaunchTimer(const char* name, cudaStream_t st) : name_(name), st_(st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  a_ = get_event();
  b_ = get_event();
  if (a_ && b_) cudaEventRecord(static_cast<cudaEvent_t>(a_), st_);
}

LaunchTimer::~LaunchTimer() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!a_ || !b_) return;
  cudaEventRecord(static_cast<cudaEvent_t>(b_), st_);
  g_pairs.push_back({name_, static_cast<cudaEvent_t>(a_), static_cast<cudaEvent_t>(b_)});
}

}  // namespace moe

extern "C" {

int moe_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(moe::g_mu);
  moe::g_on = on != 0;
  return MOE_OK;
}

int moe_timing_report(char* buf, size_t len) {
  std::lock_guard<std::mutex> lk(moe::g_mu);
  std::map<std::string, std::pair<long, double>> acc;
  for (auto& p : moe::g_pairs) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      auto& slot = acc[p.name];
      slot.first += 1;
      slot.second += ms;
    }
  }
  if (buf) {  // a report into a buffer consumes the recorded pairs
    for (auto& p : moe::g_pairs) {
      moe::g_free.push_back(p.a);
      moe::g_free.push_back(p.b);
    }
    moe::g_pairs.clear();
  }
  std::string out;
  char line[256];
  for (auto& kv : acc) {
    std::snprintf(line, sizeof(line), "%s %ld %.6f\n", kv.first.c_str(), kv.second.first,
                  kv.second.second);
    out += line;
  }
  if (buf && len) {
    std::snprintf(buf, len, "%s", out.c_str());
  }
  return static_cast<int>(out.size());
}

}  // extern "C"
