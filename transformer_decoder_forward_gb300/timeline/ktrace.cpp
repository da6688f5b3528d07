// Kernel timeline through CUPTI's activity API, loaded into a process with
// CUDA_INJECTION64_PATH: the device start and end of every kernel (also the kernels a
// replayed CUDA graph launches, and with programmatic dependent launch overlapping them),
// written at process exit as "start_ns,end_ns,grid_x,grid_y,grid_z,name" lines to the file
// named by KTRACE_OUT (default ktrace.csv).
#include <cupti.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>
#include <vector>

namespace {

struct Rec {
  std::string name;
  unsigned long long start, end;
  int gx, gy, gz;
};
std::vector<Rec> g_recs;
std::mutex g_mu;
constexpr size_t kBufferBytes = 16u << 20;
constexpr size_t kMaxRecords = 4u << 20;

void CUPTIAPI buffer_requested(uint8_t** buffer, size_t* size, size_t* max_records) {
  *size = kBufferBytes;
  *buffer = static_cast<uint8_t*>(aligned_alloc(8, kBufferBytes));
  *max_records = 0;
}

void CUPTIAPI buffer_completed(CUcontext, uint32_t, uint8_t* buffer, size_t, size_t valid) {
  CUpti_Activity* rec = nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  while (cuptiActivityGetNextRecord(buffer, valid, &rec) == CUPTI_SUCCESS) {
    if (rec->kind != CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL && rec->kind != CUPTI_ACTIVITY_KIND_KERNEL) continue;
    const auto* k = reinterpret_cast<const CUpti_ActivityKernel10*>(rec);
    if (g_recs.size() < kMaxRecords) g_recs.push_back({k->name ? k->name : "?", k->start, k->end, k->gridX, k->gridY, k->gridZ});
  }
  free(buffer);
}

void dump() {
  cuptiActivityFlushAll(1);
  const char* out = getenv("KTRACE_OUT");
  FILE* f = fopen(out ? out : "ktrace.csv", "w");
  if (!f) return;
  std::lock_guard<std::mutex> lock(g_mu);
  for (const Rec& r : g_recs) fprintf(f, "%llu,%llu,%d,%d,%d,%s\n", r.start, r.end, r.gx, r.gy, r.gz, r.name.c_str());
  fclose(f);
}

}  // namespace

extern "C" int InitializeInjection(void) {
  if (cuptiActivityRegisterCallbacks(buffer_requested, buffer_completed) != CUPTI_SUCCESS) return 0;
  if (cuptiActivityEnable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL) != CUPTI_SUCCESS) return 0;
  atexit(dump);
  return 1;
}
