// Test and tuning switches of libdh (no counterpart on the pages): which kernels serve a call.
// None of them changes results beyond the choice of kernels, and every forced path is covered by
// the GPU tests.
//
// The switches are read from the environment once per process, on first use (DH_FORCE_PATH,
// DH_FORCE_HEAD, DH_HEAD_CTAS, DH_FORCE_RESCORE, DH_SCORES_SMALL, DH_HEAD_SELECT), and can be changed afterwards
// only through dh_set_tuning, so a process's kernel choice never changes behind its back.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dh_internal.cuh"

namespace dh {
namespace {

Tuning g_tuning;
std::once_flag g_once;

// Parses one switch into t; false if the name or the value is unknown.  A null or empty value
// restores the default.
bool apply(Tuning& t, const char* name, const char* value) {
  const bool dflt = !value || !*value;
  auto is = [&](const char* v) { return !dflt && std::strcmp(value, v) == 0; };
  if (std::strcmp(name, "DH_FORCE_PATH") == 0) {
    if (dflt || is("auto")) t.force_path = Tuning::PATH_AUTO;
    else if (is("gemv")) t.force_path = Tuning::PATH_GEMV;
    else if (is("mma")) t.force_path = Tuning::PATH_MMA;
    else if (is("fused")) t.force_path = Tuning::PATH_FUSED;
    else return false;
    return true;
  }
  if (std::strcmp(name, "DH_FORCE_HEAD") == 0) {
    if (dflt || is("auto")) t.head_split = t.head_cluster = false;
    else if (is("split")) { t.head_split = true; t.head_cluster = false; }
    else if (is("cluster")) { t.head_split = false; t.head_cluster = true; }
    else return false;
    return true;
  }
  if (std::strcmp(name, "DH_HEAD_CTAS") == 0) {
    if (dflt) t.head_ctas_max = 16;
    else if (is("16")) t.head_ctas_max = 16;
    else if (is("8")) t.head_ctas_max = 8;
    else if (is("4")) t.head_ctas_max = 4;
    else if (is("2")) t.head_ctas_max = 2;
    else return false;
    return true;
  }
  if (std::strcmp(name, "DH_FORCE_RESCORE") == 0) {
    if (dflt || is("auto")) t.rescore = Tuning::RESCORE_AUTO;
    else if (is("direct")) t.rescore = Tuning::RESCORE_DIRECT;
    else if (is("ring")) t.rescore = Tuning::RESCORE_RING;
    else if (is("ticket")) t.rescore = Tuning::RESCORE_TICKET;
    else if (is("sweep")) t.rescore = Tuning::RESCORE_SWEEP;
    else if (is("bucket")) t.rescore = Tuning::RESCORE_BUCKET;  // the ring in bucket mode at any size
    else return false;
    return true;
  }
  if (std::strcmp(name, "DH_HEAD_SELECT") == 0) {
    if (dflt || is("auto") || is("fast")) t.head_select_radix = false;
    else if (is("radix")) t.head_select_radix = true;
    else return false;
    return true;
  }
  if (std::strcmp(name, "DH_SCORES_SMALL") == 0) {
    if (dflt || is("lsu")) t.scores_tma = false;
    else if (is("tma")) t.scores_tma = true;
    else return false;
    return true;
  }
  return false;
}

void init_from_env() {
  for (const char* n :
       {"DH_FORCE_PATH", "DH_FORCE_HEAD", "DH_HEAD_CTAS", "DH_FORCE_RESCORE", "DH_SCORES_SMALL", "DH_HEAD_SELECT"}) {
    Tuning t = g_tuning;
    if (apply(t, n, std::getenv(n))) g_tuning = t;  // an unknown value keeps the default
  }
}

}  // namespace

const Tuning& tuning() {
  std::call_once(g_once, init_from_env);
  return g_tuning;
}

}  // namespace dh

extern "C" int dh_set_tuning(const char* name, const char* value) {
  if (!name) return DH_ERR_INVALID_ARG;
  std::call_once(dh::g_once, dh::init_from_env);
  dh::Tuning t = dh::g_tuning;
  if (!dh::apply(t, name, value)) return DH_ERR_INVALID_ARG;
  dh::g_tuning = t;
  return DH_OK;
}
