// jit.cu -- fused kernels specialised at run time for one epilogue program.
//
// The built-in catalog covers common epilogues with straight-line kernels
// compiled with the library; any other DAG would run the interpreter.  When
// the CUDA runtime compiler (NVRTC) can be loaded, a plan instead compiles the
// same kernel template for its own program: the instruction list becomes a
// compile-time constant exactly as for a catalog entry, so the kernel is the
// catalog's straight-line code for that program, and its results are the
// interpreter's bit for bit.  The sources are the library's own headers,
// found next to the shared library; compiled kernels are kept for the life of
// the process, keyed by program and launch shape.
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "launch.h"

namespace ge {
namespace {

// the NVRTC entry points used (signatures as in nvrtc.h; handles as void *)
typedef int (*CreateProgramFn)(void **, const char *, const char *, int, const char *const *,
                               const char *const *);
typedef int (*DestroyProgramFn)(void **);
typedef int (*CompileProgramFn)(void *, int, const char *const *);
typedef int (*AddNameExpressionFn)(void *, const char *);
typedef int (*GetLoweredNameFn)(void *, const char *, const char **);
typedef int (*GetSizeFn)(void *, size_t *);
typedef int (*GetDataFn)(void *, char *);

struct Nvrtc {
  bool ok = false;
  CreateProgramFn create = nullptr;
  DestroyProgramFn destroy = nullptr;
  CompileProgramFn compile = nullptr;
  AddNameExpressionFn add_name = nullptr;
  GetLoweredNameFn lowered = nullptr;
  GetSizeFn cubin_size = nullptr, log_size = nullptr;
  GetDataFn cubin = nullptr, log = nullptr;
};

std::string cuda_home() {
  const char *h = std::getenv("CUDA_HOME");
  return h && *h ? std::string(h) : std::string("/usr/local/cuda");
}

const Nvrtc &nvrtc() {
  static Nvrtc n;
  static std::once_flag once;
  std::call_once(once, [] {
    const std::string cands[] = {"libnvrtc.so.13", "libnvrtc.so",
                                 cuda_home() + "/lib64/libnvrtc.so.13",
                                 cuda_home() + "/lib64/libnvrtc.so"};
    void *h = nullptr;
    for (const std::string &c : cands)
      if ((h = dlopen(c.c_str(), RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
    if (!h) return;
    n.create = reinterpret_cast<CreateProgramFn>(dlsym(h, "nvrtcCreateProgram"));
    n.destroy = reinterpret_cast<DestroyProgramFn>(dlsym(h, "nvrtcDestroyProgram"));
    n.compile = reinterpret_cast<CompileProgramFn>(dlsym(h, "nvrtcCompileProgram"));
    n.add_name = reinterpret_cast<AddNameExpressionFn>(dlsym(h, "nvrtcAddNameExpression"));
    n.lowered = reinterpret_cast<GetLoweredNameFn>(dlsym(h, "nvrtcGetLoweredName"));
    n.cubin_size = reinterpret_cast<GetSizeFn>(dlsym(h, "nvrtcGetCUBINSize"));
    n.cubin = reinterpret_cast<GetDataFn>(dlsym(h, "nvrtcGetCUBIN"));
    n.log_size = reinterpret_cast<GetSizeFn>(dlsym(h, "nvrtcGetProgramLogSize"));
    n.log = reinterpret_cast<GetDataFn>(dlsym(h, "nvrtcGetProgramLog"));
    n.ok = n.create && n.destroy && n.compile && n.add_name && n.lowered && n.cubin_size &&
           n.cubin && n.log_size && n.log;
  });
  return n;
}

// Directory of this shared library (…/dense_gemm_elementwise_gb300/lib).
std::string library_dir() {
  Dl_info info;
  if (!dladdr(reinterpret_cast<void *>(&library_dir), &info) || !info.dli_fname) return "";
  std::string p(info.dli_fname);
  const size_t s = p.rfind('/');
  return s == std::string::npos ? std::string(".") : p.substr(0, s);
}

std::string parent(const std::string &d) {
  const size_t s = d.rfind('/');
  return s == std::string::npos ? std::string(".") : d.substr(0, s);
}

void append_array(std::string *o, const int32_t *v, int n) {
  *o += "{";
  for (int i = 0; i < n; ++i) *o += std::to_string(v[i]) + (i + 1 < n ? "," : "");
  *o += "}";
}

void append_array(std::string *o, const uint32_t *v, int n) {
  *o += "{";
  for (int i = 0; i < n; ++i) *o += std::to_string(v[i]) + "u" + (i + 1 < n ? "," : "");
  *o += "}";
}

// The program as a constexpr aggregate (scalar values are run-time, so 0).
std::string program_literal(const EpiProgram &P) {
  std::string o = "{" + std::to_string(P.n_ins) + ",";
  append_array(&o, P.ins, kMaxIns);
  o += ",{}," + std::to_string(P.n_tma_aux) + ",";
  append_array(&o, P.tma_aux_slot, GE_MAX_TMA_AUX);
  o += ",";
  append_array(&o, P.tma_aux_dtype, GE_MAX_TMA_AUX);
  o += "," + std::to_string(P.n_bcast) + ",";
  append_array(&o, P.bcast_slot, GE_MAX_AUX);
  o += ",";
  append_array(&o, P.bcast_dtype, GE_MAX_AUX);
  o += "," + std::to_string(P.n_cbcast) + ",";
  append_array(&o, P.cbcast_slot, GE_MAX_AUX);
  o += ",";
  append_array(&o, P.cbcast_dtype, GE_MAX_AUX);
  o += "," + std::to_string(P.n_out) + ",";
  append_array(&o, P.out_dtype, GE_MAX_OUT);
  o += "," + std::to_string(P.n_regs) + "}";
  return o;
}

std::string cache_key(const EpiProgram &P, int cg, int bn, int warps) {
  std::string k = program_literal(P);
  k += "|" + std::to_string(cg) + "," + std::to_string(bn) + "," + std::to_string(warps);
  return k;
}

std::mutex g_jit_mutex;
std::map<std::string, const void *> g_jit_cache;

}  // namespace

bool jit_available() { return nvrtc().ok; }

const void *jit_gemm_kernel(const EpiProgram &P, int cg, int bn, int warps, std::string *log) {
  const Nvrtc &n = nvrtc();
  if (!n.ok) {
    if (log) *log = "runtime compiler (libnvrtc) not found";
    return nullptr;
  }
  const std::string key = cache_key(P, cg, bn, warps);
  std::lock_guard<std::mutex> lock(g_jit_mutex);
  auto it = g_jit_cache.find(key);
  if (it != g_jit_cache.end()) return it->second;

  const std::string lib = library_dir();
  const std::string csrc = parent(lib) + "/csrc";
  const std::string inc = parent(parent(lib)) + "/include";
  const std::string src = "#include \"gemm_kernel.cuh\"\n"
                          "namespace ge {\n"
                          "struct JitProg {\n"
                          "  static constexpr EpiProgram P = " +
                          program_literal(P) +
                          ";\n"
                          "};\n"
                          "}  // namespace ge\n";
  const std::string name = "ge::gemm_epi_kernel<" + std::to_string(cg) + ", " +
                           std::to_string(bn) + ", ge::EpiStatic<ge::JitProg, " + std::to_string(warps) + "> >";
  const std::string o_csrc = "-I" + csrc, o_inc = "-I" + inc,
                    o_cuda = "-I" + cuda_home() + "/include";
  // -default-device: the C ABI's host declarations in gemm_epi.h are never
  // used by the kernel, which the compiler otherwise refuses in this mode
  const char *opts[] = {"-arch=sm_103a", "-std=c++17", "-default-device", "-DNDEBUG",
                        o_csrc.c_str(), o_inc.c_str(), o_cuda.c_str()};

  void *prog = nullptr;
  const void *fn = nullptr;
  std::string errlog;
  if (n.create(&prog, src.c_str(), "gemm_epi_jit.cu", 0, nullptr, nullptr) == 0 &&
      n.add_name(prog, name.c_str()) == 0) {
    const int cr = n.compile(prog, static_cast<int>(sizeof(opts) / sizeof(opts[0])), opts);
    size_t ls = 0;
    if (n.log_size(prog, &ls) == 0 && ls > 1) {
      errlog.resize(ls);
      n.log(prog, &errlog[0]);
    }
    const char *lowered = nullptr;
    size_t cs = 0;
    if (cr == 0 && n.lowered(prog, name.c_str(), &lowered) == 0 && lowered &&
        n.cubin_size(prog, &cs) == 0 && cs > 0) {
      std::vector<char> cubin(cs);
      cudaLibrary_t libh = nullptr;
      cudaKernel_t kern = nullptr;
      if (n.cubin(prog, cubin.data()) == 0 &&
          cudaLibraryLoadData(&libh, cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0) ==
              cudaSuccess &&
          cudaLibraryGetKernel(&kern, libh, lowered) == cudaSuccess)
        fn = reinterpret_cast<const void *>(kern);
      cudaGetLastError();
    }
    n.destroy(&prog);
  }
  if (log) *log = errlog;
  if (fn) g_jit_cache[key] = fn;
  return fn;
}

}  // namespace ge
