// Per-shape choice of the bf16 forward kernel: a process-wide table from a
// problem class to (kernel, raster), filled by gmm_tune() or gmm_tuning_set()
// and kept in a text file by gmm_tuning_save() / gmm_tuning_load().
//
// The pages let `tiling` be a callable that looks the problem dimensions up in a
// LUT of tuned tile sizes (page "tpu-inference 0.12.0.dev20251213 ->
// 0.13.2.dev20251230", gmm.py: "If tiling is callable, look up the problem
// dimensions in the LUT").  Here the tiles of each kernel are fixed; what varies
// per problem is which of the four bf16 kernels runs and, for the row-tile
// kernels, the order of their tiles (how many n tiles share a super-column of
// the L2 raster, or, negative, how many m tiles of a group form a block that
// meets every n tile in turn).  m changes
// with routing, so the table keys on floor(log2(m / num_total_groups)), the
// average rows per group, next to k, n, the group count, the layout and the
// output dtype.
//
// File format: a first line "# libgmm tiling table 1", then one entry per line,
//   rows_log2 k n num_total_groups transpose_rhs out_dtype kernel raster
// as decimal integers separated by blanks; blank lines and lines starting with
// '#' are skipped.
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/libgmm.h"
#include "internal.h"

namespace gmmk {
namespace {

using Key = std::tuple<int32_t, int64_t, int64_t, int32_t, int32_t, int32_t>;
struct Choice {
  int32_t kernel;
  int32_t raster;
};

std::mutex g_lock;
std::map<Key, Choice>& table() {
  static std::map<Key, Choice> t;
  return t;
}

constexpr const char* kHeader = "# libgmm tiling table 1";

}  // namespace

int32_t tuning_rows_log2(int64_t m, int32_t num_total_groups) {
  int64_t avg = num_total_groups > 0 ? m / num_total_groups : m;
  int32_t l = 0;
  while (avg > 1) {
    avg >>= 1;
    ++l;
  }
  return l;
}

bool tuning_lookup(int32_t rows_log2, int64_t k, int64_t n, int32_t groups, int32_t transpose, int32_t out_dtype,
                   int32_t* kernel, int32_t* raster) {
  std::lock_guard<std::mutex> g(g_lock);
  auto it = table().find(Key{rows_log2, k, n, groups, transpose, out_dtype});
  if (it == table().end()) return false;
  *kernel = it->second.kernel;
  *raster = it->second.raster;
  return true;
}

void tuning_store(int32_t rows_log2, int64_t k, int64_t n, int32_t groups, int32_t transpose, int32_t out_dtype,
                  int32_t kernel, int32_t raster) {
  std::lock_guard<std::mutex> g(g_lock);
  table()[Key{rows_log2, k, n, groups, transpose, out_dtype}] = Choice{kernel, raster};
}

bool tuning_valid(int32_t kernel, int32_t raster) {
  return kernel >= GMM_KERNEL_PAIR && kernel <= GMM_KERNEL_SINGLE && raster >= -64 && raster <= 64;
}

}  // namespace gmmk

extern "C" {

int gmm_tuning_set(int32_t rows_log2, int64_t k, int64_t n, int32_t num_total_groups, int transpose_rhs,
                   int out_dtype, int kernel, int raster) {
  if (rows_log2 < 0 || rows_log2 > 62 || k < 1 || n < 1 || num_total_groups < 1) return GMM_ERR_SHAPE;
  if (!gmmk::tuning_valid(kernel, raster)) return GMM_ERR_SHAPE;
  gmmk::tuning_store(rows_log2, k, n, num_total_groups, transpose_rhs != 0, out_dtype, kernel, raster);
  return GMM_OK;
}

int gmm_tuning_get(int32_t rows_log2, int64_t k, int64_t n, int32_t num_total_groups, int transpose_rhs,
                   int out_dtype, int* kernel, int* raster) {
  if (kernel == nullptr || raster == nullptr) return GMM_ERR_NULL;
  int32_t kk = GMM_KERNEL_AUTO, rr = 0;
  gmmk::tuning_lookup(rows_log2, k, n, num_total_groups, transpose_rhs != 0, out_dtype, &kk, &rr);
  *kernel = kk;
  *raster = rr;
  return GMM_OK;
}

int gmm_tuning_clear(void) {
  std::lock_guard<std::mutex> g(gmmk::g_lock);
  gmmk::table().clear();
  return GMM_OK;
}

int gmm_tuning_save(const char* path) {
  if (path == nullptr) return GMM_ERR_NULL;
  std::FILE* f = std::fopen(path, "w");
  if (f == nullptr) return GMM_ERR_IO;
  bool ok = std::fprintf(f, "%s\n", gmmk::kHeader) > 0;
  {
    std::lock_guard<std::mutex> g(gmmk::g_lock);
    for (const auto& [key, c] : gmmk::table()) {
      ok = ok && std::fprintf(f, "%d %lld %lld %d %d %d %d %d\n", std::get<0>(key),
                              static_cast<long long>(std::get<1>(key)), static_cast<long long>(std::get<2>(key)),
                              std::get<3>(key), std::get<4>(key), std::get<5>(key), c.kernel, c.raster) > 0;
    }
  }
  ok = (std::fclose(f) == 0) && ok;
  return ok ? GMM_OK : GMM_ERR_IO;
}

int gmm_tuning_load(const char* path) {
  if (path == nullptr) return GMM_ERR_NULL;
  std::FILE* f = std::fopen(path, "r");
  if (f == nullptr) return GMM_ERR_IO;
  char line[512];
  bool ok = std::fgets(line, sizeof line, f) != nullptr && std::strncmp(line, gmmk::kHeader, std::strlen(gmmk::kHeader)) == 0;
  struct Entry {
    int rows_log2, groups, transpose, out_dtype, kernel, raster;
    long long k, n;
  };
  Entry e{};
  std::map<gmmk::Key, gmmk::Choice> loaded;
  while (ok && std::fgets(line, sizeof line, f) != nullptr) {
    const char* c = line;
    while (*c == ' ' || *c == '\t') ++c;
    if (*c == '#' || *c == '\n' || *c == '\r' || *c == '\0') continue;
    char tail = 0;
    const int got = std::sscanf(c, "%d %lld %lld %d %d %d %d %d %c", &e.rows_log2, &e.k, &e.n, &e.groups, &e.transpose,
                                &e.out_dtype, &e.kernel, &e.raster, &tail);
    if (got != 8 || e.rows_log2 < 0 || e.rows_log2 > 62 || e.k < 1 || e.n < 1 || e.groups < 1 ||
        !gmmk::tuning_valid(e.kernel, e.raster)) {
      ok = false;
      break;
    }
    loaded[gmmk::Key{e.rows_log2, e.k, e.n, e.groups, e.transpose != 0, e.out_dtype}] = gmmk::Choice{e.kernel, e.raster};
  }
  std::fclose(f);
  if (!ok) return GMM_ERR_IO;
  std::lock_guard<std::mutex> g(gmmk::g_lock);
  for (const auto& [key, c] : loaded) gmmk::table()[key] = c;
  return GMM_OK;
}

}  // extern "C"
