// route_trace.cu -- expert usage history files (host code only).
//
// The format is the one the colibri tuning guide describes for its usage
// history (gitcode.com colibri tuning guide, "usage-history format",
// route_trace.h): text, one record per line, sparse.  Two header records carry
// the dimensions (-1 n_layers n_experts) and the writer's identity
// (-2 format_version engine_id); every other record is layer expert count for
// a non-zero count.  The guide's constraints, and how they shape this code:
//   - every field is a number, and a record has exactly three of them: a
//     string or a fourth field would make a scanf-style reader lose its place;
//   - the engine is named by its FNV-1a 32-bit hash, which can exceed
//     INT_MAX, so it sits in the third field with the small version second;
//   - readers skip any record whose first field is negative, so header types
//     can be added later without breaking older readers;
//   - an empty history is a zero-byte file, with no header.
// The guide gives no version number; this writer uses 1.  The reader also
// accepts the older headerless form (triplets only).
#include <errno.h>
#include <stdio.h>
#include <stdlib.h>

#include <vector>

#include "moe_internal.cuh"

namespace {

constexpr long long kFormatVersion = 1;

// Splits one line into integer fields; false if a field is not an integer or
// there are not exactly three of them.
bool parse_record(const char *p, const char *end, long long f[3]) {
  int n = 0;
  while (p < end) {
    while (p < end && (*p == ' ' || *p == '\t' || *p == '\r')) ++p;
    if (p == end) break;
    if (n == 3) return false;
    const char *q = p;
    if (*q == '-' || *q == '+') ++q;
    if (q == end || *q < '0' || *q > '9') return false;
    while (q < end && *q >= '0' && *q <= '9') ++q;
    if (q < end && *q != ' ' && *q != '\t' && *q != '\r') return false;
    char buf[32];
    const size_t len = (size_t)(q - p);
    if (len >= sizeof(buf)) return false;
    for (size_t i = 0; i < len; ++i) buf[i] = p[i];
    buf[len] = 0;
    errno = 0;
    f[n++] = strtoll(buf, nullptr, 10);
    if (errno) return false;
    p = q;
  }
  return n == 3;
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) uint32_t moe_engine_id(const char *name) {
  if (!name) return 0;
  uint32_t hash = 2166136261u;
  for (const unsigned char *c = reinterpret_cast<const unsigned char *>(name); *c; ++c) {
    hash ^= *c;
    hash *= 16777619u;
  }
  return hash;
}

__attribute__((visibility("default"))) int moe_route_trace_write(const char *path, int n_layers,
                                                                 int n_experts, uint32_t engine_id,
                                                                 const int64_t *counts) {
  if (!path || !counts || n_layers < 1 || n_experts < 1) return MOE_ERR_ARG;
  const size_t n = (size_t)n_layers * n_experts;
  bool any = false;
  for (size_t i = 0; i < n; ++i) {
    if (counts[i] < 0) return MOE_ERR_ARG;
    any = any || counts[i] > 0;
  }
  FILE *f = fopen(path, "wb");
  if (!f) return MOE_ERR_IO;
  bool ok = true;
  if (any) {
    ok = fprintf(f, "-1 %d %d\n-2 %lld %u\n", n_layers, n_experts, kFormatVersion,
                 (unsigned)engine_id) > 0;
    for (int l = 0; ok && l < n_layers; ++l)
      for (int e = 0; ok && e < n_experts; ++e) {
        const long long c = counts[(size_t)l * n_experts + e];
        if (c) ok = fprintf(f, "%d %d %lld\n", l, e, c) > 0;
      }
  }
  ok = (fclose(f) == 0) && ok;
  return ok ? MOE_OK : MOE_ERR_IO;
}

__attribute__((visibility("default"))) int moe_route_trace_read(const char *path, int n_layers,
                                                                int n_experts, uint32_t engine_id,
                                                                int64_t *counts,
                                                                uint32_t *found_engine) {
  if (!path || !counts || n_layers < 1 || n_experts < 1) return MOE_ERR_ARG;
  if (found_engine) *found_engine = 0;
  FILE *f = fopen(path, "rb");
  if (!f) return MOE_ERR_IO;
  std::vector<char> text;
  char chunk[1 << 16];
  size_t got;
  while ((got = fread(chunk, 1, sizeof(chunk), f)) > 0) text.insert(text.end(), chunk, chunk + got);
  const bool read_err = ferror(f) != 0;
  fclose(f);
  if (read_err) return MOE_ERR_IO;
  if (text.empty()) return MOE_OK;   // empty history

  std::vector<int64_t> add((size_t)n_layers * n_experts, 0);
  uint32_t engine = 0;
  bool dims_bad = false, engine_bad = false;
  const char *p = text.data(), *end = p + text.size();
  while (p < end) {
    const char *eol = p;
    while (eol < end && *eol != '\n') ++eol;
    const char *q = p;
    while (q < eol && (*q == ' ' || *q == '\t' || *q == '\r')) ++q;
    if (q < eol) {   // blank lines carry no record
      long long r[3];
      if (!parse_record(p, eol, r)) return MOE_ERR_IO;
      if (r[0] < 0) {
        if (r[0] == -1 && (r[1] != n_layers || r[2] != n_experts)) dims_bad = true;
        if (r[0] == -2) {
          if (r[2] < 0 || r[2] > 0xffffffffLL) return MOE_ERR_IO;
          engine = (uint32_t)r[2];
          if (engine_id != 0 && engine != engine_id) engine_bad = true;
        }
        // any other negative record type: a header this reader does not know
      } else {
        if (r[0] >= n_layers || r[1] < 0 || r[1] >= n_experts || r[2] < 0) return MOE_ERR_IO;
        add[(size_t)r[0] * n_experts + r[1]] += r[2];
      }
    }
    p = eol < end ? eol + 1 : end;
  }
  if (found_engine) *found_engine = engine;
  if (dims_bad || engine_bad) return MOE_ERR_ENGINE;
  for (size_t i = 0; i < add.size(); ++i) counts[i] += add[i];
  return MOE_OK;
}

}  // extern "C"
