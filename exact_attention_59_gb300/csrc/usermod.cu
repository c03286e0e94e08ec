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
//
// A user mask_mod (create_block_mask takes any mask function in the
// flaxattention README) is a second C expression, nonzero = keep; it is
// compiled into the same kernels (evaluated on the entries of PARTIAL tiles of
// a block mask whose mask_mod is ATTN_MASKMOD_USER) and into a block-mask
// builder (usermask.cuh) that gives the tile states.
#include <dlfcn.h>
#include <nvrtc.h>

#include <algorithm>
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
  bool has_mask;
  std::vector<char> cubin;
  std::string names[4];   // lowered names: forward, dK/dV, dQ, block-mask builder (with a mask)
  std::mutex mu;
  struct Loaded {
    cudaLibrary_t lib;
    cudaKernel_t k[4];
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

extern "C" attn_status attn_user_mod_create_masked(const char* bias_expr, const char* mask_expr, attn_dtype dtype,
                                                   attn_user_mod* mod, char* log, size_t log_bytes) {
  if (!mod) return ATTN_ERR_INVALID_ARG;
  *mod = nullptr;
  const size_t blen = bias_expr ? std::strlen(bias_expr) : 0, mlen = mask_expr ? std::strlen(mask_expr) : 0;
  if ((blen == 0 && mlen == 0) || blen > 4096 || mlen > 4096) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  const std::string dir = csrc_dir();
  if (FILE* f = std::fopen((dir + "/fwd_d64.cu").c_str(), "r")) {
    std::fclose(f);
  } else {
    put_log(log, log_bytes, "kernel sources not found in " + dir);
    return ATTN_ERR_UNSUPPORTED;
  }
  const bool has_mask = mlen > 0;
  std::string src = "#define ATTN_USER_BIAS_EXPR (" + std::string(blen ? bias_expr : "0.0f") + ")\n";
  if (has_mask) src += "#define ATTN_USER_MASK_EXPR (" + std::string(mask_expr) + ")\n";
  src += "#include \"fwd_d64.cu\"\n#include \"bwd_d64.cu\"\n";
  if (has_mask) src += "#include \"usermask.cuh\"\n";
  const char* bf = dtype == ATTN_BF16 ? "true" : "false";
  const std::string exprs[4] = {std::string("attn::fwd_d64_kernel<") + bf + ", 4, 0>",
                                std::string("attn::bwd_dkdv_kernel<") + bf + ", 4, false>",
                                std::string("attn::bwd_dq_kernel<") + bf + ", 4, false>",
                                std::string("attn::user_block_mask_kernel")};
  const int nk = has_mask ? 4 : 3;
  nvrtcProgram prog;
  if (nvrtcCreateProgram(&prog, src.c_str(), "user_score_mod.cu", 0, nullptr, nullptr) != NVRTC_SUCCESS)
    return ATTN_ERR_CUDA;
  for (int i = 0; i < nk; ++i) nvrtcAddNameExpression(prog, exprs[i].c_str());
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
    return ATTN_ERR_INVALID_ARG;   // an expression does not compile: the log says why
  }
  attn_user_mod m = new attn_user_mod_st();
  m->dtype = dtype;
  m->has_mask = has_mask;
  size_t n = 0;
  nvrtcGetCUBINSize(prog, &n);
  m->cubin.resize(n);
  nvrtcGetCUBIN(prog, m->cubin.data());
  for (int i = 0; i < nk; ++i) {
    const char* lowered = nullptr;
    nvrtcGetLoweredName(prog, exprs[i].c_str(), &lowered);
    m->names[i] = lowered ? lowered : "";
  }
  nvrtcDestroyProgram(&prog);
  *mod = m;
  return ATTN_OK;
}

extern "C" attn_status attn_user_mod_create(const char* bias_expr, attn_dtype dtype, attn_user_mod* mod, char* log,
                                            size_t log_bytes) {
  if (!bias_expr || !mod || bias_expr[0] == '\0') return ATTN_ERR_INVALID_ARG;
  return attn_user_mod_create_masked(bias_expr, nullptr, dtype, mod, log, log_bytes);
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

namespace {

// The mod's kernels on the current device (its code loaded there on first use).
attn_status loaded_kernels(attn_user_mod mod, const void* (&kern)[4]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  const int nk = mod->has_mask ? 4 : 3;
  std::lock_guard<std::mutex> g(mod->mu);
  auto it = mod->per_device.find(dev);
  if (it == mod->per_device.end()) {
    attn_user_mod_st::Loaded L{};
    if (cudaLibraryLoadData(&L.lib, mod->cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    for (int i = 0; i < nk; ++i) {
      if (cudaLibraryGetKernel(&L.k[i], L.lib, mod->names[i].c_str()) != cudaSuccess) {
        cudaLibraryUnload(L.lib);
        return ATTN_ERR_CUDA;
      }
    }
    it = mod->per_device.emplace(dev, L).first;
  }
  for (int i = 0; i < 4; ++i) kern[i] = i < nk ? reinterpret_cast<const void*>(it->second.k[i]) : nullptr;
  return ATTN_OK;
}

}  // namespace

attn_status user_mod_kernels(attn_user_mod mod, attn_dtype dtype, const void* (&kern)[3]) {
  if (!mod) return ATTN_ERR_INVALID_ARG;
  if (mod->dtype != dtype) return ATTN_ERR_UNSUPPORTED;   // built for the other 16-bit type
  const void* all[4];
  const attn_status st = loaded_kernels(mod, all);
  if (st != ATTN_OK) return st;
  for (int i = 0; i < 3; ++i) kern[i] = all[i];
  return ATTN_OK;
}

bool user_mod_has_mask(attn_user_mod mod) { return mod && mod->has_mask; }

}  // namespace attn

extern "C" attn_status attn_build_block_mask_user(attn_user_mod mod, int B, int H, int Sq, int Skv, int bq, int bkv,
                                                  uint8_t* tiles, attn_stream_t stream) {
  using namespace attn;
  if (!mod || !mod->has_mask || !tiles || B <= 0 || H <= 0 || Sq <= 0 || Skv <= 0 || bq <= 0 || bkv <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (bq != 128 || bkv != 128) return ATTN_ERR_UNSUPPORTED;
  const void* kern[4];
  const attn_status st = loaded_kernels(mod, kern);
  if (st != ATTN_OK) return st;
  const long long ntiles = (long long)B * H * ((Sq + 127) / 128) * ((Skv + 127) / 128);
  const unsigned grid = (unsigned)std::min<long long>(ntiles, 152LL * 16);
  void* args[] = {&B, &H, &Sq, &Skv, &tiles};
  return cudaLaunchKernel(kern[3], dim3(grid), dim3(256), args, 0, (cudaStream_t)stream) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}
