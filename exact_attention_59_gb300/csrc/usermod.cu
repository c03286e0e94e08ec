// usermod.cu - score_mods compiled at run time (NVRTC) into the D = 64 kernels.
//
// The flaxattention README's hooks take arbitrary callables (score_mod(score,
// b, h, q_idx, kv_idx)); the built-in enum covers the ones it names.  A user
// score_mod here is a C expression for an additive bias in the variables b, h,
// q and kv (int; q and kv are positions), -INFINITY to mask: every mod the
// pages name is of this form, so d score' / d score = 1 and the recompute
// backward needs nothing else.  The expression is compiled into the same
// forward, dK/dV and dQ kernel sources as the built-in mods (as the MOD_USER
// instantiation), so the generated kernels have the built-in ones' layout,
// pipelines and bounded waits.  Compilation needs no GPU; the cubin is loaded
// on a device the first time a call on that device uses it.
#include <dlfcn.h>
#include <nvrtc.h>

#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/attn.h"
#include "kernels.h"
#include "usermod.h"

struct attn_user_mod_st {
  attn_dtype dtype;
  std::vector<char> cubin;
  std::string names[3];   // lowered names: forward, dK/dV, dQ
  std::mutex mu;
  struct Loaded {
    cudaLibrary_t lib;
    cudaKernel_t k[3];
  };
  std::map<int, Loaded> per_device;
};

namespace {

// The kernel sources sit in csrc/ beside the shared library.
std::string csrc_dir() {
  Dl_info info;
  if (!dladdr(reinterpret_cast<void*>(&attn_user_mod_create), &info) || !info.dli_fname) return "";
  std::string p(info.dli_fname);
  const size_t slash = p.rfind('/');
  return (slash == std::string::npos ? std::string(".") : p.substr(0, slash)) + "/csrc";
}

void put_log(char* log, size_t log_bytes, const std::string& text) {
  if (!log || log_bytes == 0) return;
  const size_t n = std::min(log_bytes - 1, text.size());
  std::memcpy(log, text.data(), n);
  log[n] = '\0';
}

}  // namespace

extern "C" attn_status attn_user_mod_create(const char* bias_expr, attn_dtype dtype, attn_user_mod* mod, char* log,
                                            size_t log_bytes) {
  if (!bias_expr || !mod) return ATTN_ERR_INVALID_ARG;
  *mod = nullptr;
  const size_t len = std::strlen(bias_expr);
  if (len == 0 || len > 4096) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  const std::string dir = csrc_dir();
  if (FILE* f = std::fopen((dir + "/fwd_d64.cu").c_str(), "r")) {
    std::fclose(f);
  } else {
    put_log(log, log_bytes, "kernel sources not found in " + dir);
    return ATTN_ERR_UNSUPPORTED;
  }
  const std::string src = "#define ATTN_USER_BIAS_EXPR (" + std::string(bias_expr) +
                          ")\n#include \"fwd_d64.cu\"\n#include \"bwd_d64.cu\"\n";
  const char* bf = dtype == ATTN_BF16 ? "true" : "false";
  const std::string exprs[3] = {std::string("attn::fwd_d64_kernel<") + bf + ", 4, 0>",
                                std::string("attn::bwd_dkdv_kernel<") + bf + ", 4, false>",
                                std::string("attn::bwd_dq_kernel<") + bf + ", 4, false>"};
  nvrtcProgram prog;
  if (nvrtcCreateProgram(&prog, src.c_str(), "user_score_mod.cu", 0, nullptr, nullptr) != NVRTC_SUCCESS)
    return ATTN_ERR_CUDA;
  for (const std::string& e : exprs) nvrtcAddNameExpression(prog, e.c_str());
  const std::string inc = "-I" + dir;
  // -default-device: the kernels' lambdas carry no execution-space annotation
  const char* opts[] = {"--gpu-architecture=sm_103a", "-std=c++17", "-default-device", inc.c_str()};
  const nvrtcResult rc = nvrtcCompileProgram(prog, 4, opts);
  size_t log_size = 0;
  nvrtcGetProgramLogSize(prog, &log_size);
  std::string text(log_size, '\0');
  if (log_size) nvrtcGetProgramLog(prog, &text[0]);
  put_log(log, log_bytes, text);
  if (rc != NVRTC_SUCCESS) {
    nvrtcDestroyProgram(&prog);
    return ATTN_ERR_INVALID_ARG;   // the expression does not compile: the log says why
  }
  attn_user_mod m = new attn_user_mod_st();
  m->dtype = dtype;
  size_t n = 0;
  nvrtcGetCUBINSize(prog, &n);
  m->cubin.resize(n);
  nvrtcGetCUBIN(prog, m->cubin.data());
  for (int i = 0; i < 3; ++i) {
    const char* lowered = nullptr;
    nvrtcGetLoweredName(prog, exprs[i].c_str(), &lowered);
    m->names[i] = lowered ? lowered : "";
  }
  nvrtcDestroyProgram(&prog);
  *mod = m;
  return ATTN_OK;
}

extern "C" void attn_user_mod_destroy(attn_user_mod mod) {
  if (!mod) return;
  // Kernels of this mod may still be queued (calls are asynchronous): each
  // device it was loaded on finishes its work before the code is unloaded.
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : mod->per_device) {
    if (cudaSetDevice(kv.first) == cudaSuccess) cudaDeviceSynchronize();
    cudaLibraryUnload(kv.second.lib);
  }
  if (have_cur) cudaSetDevice(cur);
  delete mod;
}

namespace attn {

attn_status user_mod_kernels(attn_user_mod mod, attn_dtype dtype, const void* (&kern)[3]) {
  if (!mod) return ATTN_ERR_INVALID_ARG;
  if (mod->dtype != dtype) return ATTN_ERR_UNSUPPORTED;   // built for the other 16-bit type
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> g(mod->mu);
  auto it = mod->per_device.find(dev);
  if (it == mod->per_device.end()) {
    attn_user_mod_st::Loaded L;
    if (cudaLibraryLoadData(&L.lib, mod->cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    for (int i = 0; i < 3; ++i) {
      if (cudaLibraryGetKernel(&L.k[i], L.lib, mod->names[i].c_str()) != cudaSuccess) {
        cudaLibraryUnload(L.lib);
        return ATTN_ERR_CUDA;
      }
    }
    it = mod->per_device.emplace(dev, L).first;
  }
  for (int i = 0; i < 3; ++i) kern[i] = reinterpret_cast<const void*>(it->second.k[i]);
  return ATTN_OK;
}

}  // namespace attn
