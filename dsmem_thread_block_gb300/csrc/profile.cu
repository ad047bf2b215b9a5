// profile.cu -- the persisted calibration profile and the planning switches.
//
// The cost model's inputs that cost time to measure -- the DSMEM profile
// (cluster barrier, replicated push and st.async exchange per cluster size)
// and the plan it chose per shape after timing candidates -- are written to
// a JSON file and read back by later processes, so they plan without
// recalibrating or re-tuning.  A profile is tied to what produced it: the GPU
// name, SM count, peak SM and memory clocks, compute capability and the
// library version; a profile whose key differs from the device it is loaded
// on is stale and is rejected (the caller recalibrates).  Plans read back are
// re-derived on the loading device, so a profile can never launch an illegal
// configuration.
//
//   CREDIT_PROFILE=<path>   load <path> at the first planning call on each
//                           device, and write the state back after every
//                           calibration or profiled plan
//   CREDIT_FORCE=<plan>     the automatic plan of every shape becomes <plan>
//                           where it is legal: cluster:P[xR][:sN] (N: staged
//                           elements of an L2-tail plan), persist:P, pipe:P,
//                           warp_rows, twopass
#include <cuda_runtime.h>

#include <cctype>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "credit.h"
#include "common.cuh"
#include "internal.h"
#include "planner.h"

namespace credit {
namespace {

constexpr const char* kFormat = "credit-profile-1";

// ------------------------------------------------------------ JSON reader
// Enough JSON for the profile: objects, arrays, strings, numbers, literals;
// nesting is bounded so a hostile file cannot exhaust the stack.
struct Json {
    enum Kind { kNull, kBool, kNum, kStr, kArr, kObj } kind = kNull;
    double num = 0.0;
    bool b = false;
    std::string str;
    std::vector<Json> arr;
    std::vector<std::pair<std::string, Json>> obj;
    const Json* get(const char* key) const {
        if (kind != kObj) return nullptr;
        for (const auto& kv : obj)
            if (kv.first == key) return &kv.second;
        return nullptr;
    }
};

struct Parser {
    const char* p;
    const char* end;
    bool ok = true;
    int depth = 0;

    void ws() {
        while (p < end && std::isspace((unsigned char)*p)) ++p;
    }
    bool lit(const char* s) {
        const size_t n = std::strlen(s);
        if ((size_t)(end - p) >= n && std::memcmp(p, s, n) == 0) {
            p += n;
            return true;
        }
        return false;
    }
    bool string(std::string* out) {
        if (p >= end || *p != '"') return false;
        ++p;
        while (p < end && *p != '"') {
            char c = *p++;
            if (c == '\\') {
                if (p >= end) return false;
                const char e = *p++;
                switch (e) {
                    case 'n': c = '\n'; break;
                    case 't': c = '\t'; break;
                    case 'r': c = '\r'; break;
                    case 'b': c = '\b'; break;
                    case 'f': c = '\f'; break;
                    case 'u':  // kept as '?': the profile writes no escapes of this kind
                        if (end - p < 4) return false;
                        p += 4;
                        c = '?';
                        break;
                    default: c = e;  // \" \\ \/
                }
            }
            out->push_back(c);
        }
        if (p >= end) return false;
        ++p;
        return true;
    }
    Json value() {
        Json v;
        ws();
        if (!ok || p >= end || ++depth > 32) {
            ok = false;
            return v;
        }
        const char c = *p;
        if (c == '{') {
            ++p;
            v.kind = Json::kObj;
            ws();
            if (p < end && *p == '}') {
                ++p;
            } else {
                for (;;) {
                    ws();
                    std::string k;
                    if (!string(&k)) { ok = false; break; }
                    ws();
                    if (p >= end || *p != ':') { ok = false; break; }
                    ++p;
                    Json item = value();
                    if (!ok) break;
                    v.obj.emplace_back(std::move(k), std::move(item));
                    ws();
                    if (p < end && *p == ',') { ++p; continue; }
                    if (p < end && *p == '}') { ++p; break; }
                    ok = false;
                    break;
                }
            }
        } else if (c == '[') {
            ++p;
            v.kind = Json::kArr;
            ws();
            if (p < end && *p == ']') {
                ++p;
            } else {
                for (;;) {
                    Json item = value();
                    if (!ok) break;
                    v.arr.push_back(std::move(item));
                    ws();
                    if (p < end && *p == ',') { ++p; continue; }
                    if (p < end && *p == ']') { ++p; break; }
                    ok = false;
                    break;
                }
            }
        } else if (c == '"') {
            v.kind = Json::kStr;
            if (!string(&v.str)) ok = false;
        } else if (lit("true")) {
            v.kind = Json::kBool;
            v.b = true;
        } else if (lit("false")) {
            v.kind = Json::kBool;
        } else if (lit("null")) {
            v.kind = Json::kNull;
        } else {
            char buf[64];
            size_t n = 0;
            while (p < end && n < sizeof(buf) - 1 &&
                   (std::isdigit((unsigned char)*p) || *p == '-' || *p == '+' || *p == '.' ||
                    *p == 'e' || *p == 'E'))
                buf[n++] = *p++;
            buf[n] = 0;
            char* stop = nullptr;
            v.num = std::strtod(buf, &stop);
            v.kind = Json::kNum;
            if (n == 0 || stop != buf + n) ok = false;
        }
        --depth;
        return v;
    }
};

bool read_file(const char* path, std::string* out) {
    FILE* f = std::fopen(path, "rb");
    if (!f) return false;
    char buf[65536];
    size_t n;
    while ((n = std::fread(buf, 1, sizeof(buf), f)) > 0) {
        out->append(buf, n);
        if (out->size() > ((size_t)64 << 20)) break;  // no profile is this large
    }
    std::fclose(f);
    return out->size() <= ((size_t)64 << 20);
}

bool parse(const std::string& text, Json* out) {
    Parser ps{text.data(), text.data() + text.size()};
    *out = ps.value();
    ps.ws();
    return ps.ok && ps.p == ps.end && out->kind == Json::kObj;
}

// ------------------------------------------------------------- device key
bool device_key(int dev, credit_device_key_t* k) {
    std::memset(k, 0, sizeof(*k));
    cudaDeviceProp prop;
    int sm_khz = 0, mem_khz = 0;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_khz, cudaDevAttrClockRate, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&mem_khz, cudaDevAttrMemoryClockRate, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::snprintf(k->gpu_name, sizeof(k->gpu_name), "%s", prop.name);
    k->sms = prop.multiProcessorCount;
    k->sm_clock_mhz = sm_khz / 1000;
    k->mem_clock_mhz = mem_khz / 1000;
    k->cc_major = prop.major;
    k->cc_minor = prop.minor;
    return true;
}

double num_or(const Json* j, double dflt) {
    return j && j->kind == Json::kNum ? j->num : dflt;
}

// OK: the profile belongs to `key` and this library; NOT_CALIBRATED: a
// readable profile of another device, clock setting or library version
// (stale); INVALID_ARG: not a profile.
credit_status_t check(const Json& root, const credit_device_key_t& key) {
    const Json* fmt = root.get("format");
    const Json* lib = root.get("library");
    const Json* dev = root.get("device");
    if (!fmt || fmt->kind != Json::kStr || fmt->str != kFormat || !lib || lib->kind != Json::kStr ||
        !dev || dev->kind != Json::kObj)
        return CREDIT_ERR_INVALID_ARG;
    const Json* name = dev->get("name");
    if (!name || name->kind != Json::kStr) return CREDIT_ERR_INVALID_ARG;
    if (lib->str != credit_version()) return CREDIT_ERR_NOT_CALIBRATED;
    if (name->str != key.gpu_name || num_or(dev->get("sms"), -1) != key.sms ||
        num_or(dev->get("sm_clock_mhz"), -1) != key.sm_clock_mhz ||
        num_or(dev->get("mem_clock_mhz"), -1) != key.mem_clock_mhz ||
        num_or(dev->get("cc_major"), -1) != key.cc_major ||
        num_or(dev->get("cc_minor"), -1) != key.cc_minor)
        return CREDIT_ERR_NOT_CALIBRATED;
    return CREDIT_OK;
}

// JSON string body of `s` (the device name is the only free text written).
std::string escaped(const char* s) {
    std::string o;
    for (; *s; ++s) {
        const unsigned char c = (unsigned char)*s;
        if (c == '"' || c == '\\') {
            o.push_back('\\');
            o.push_back((char)c);
        } else if (c >= 0x20) {
            o.push_back((char)c);
        }
    }
    return o;
}

// The plan fields a profile stores, in this order.
constexpr int kPlanFields = 16;

void plan_to_array(const credit_plan_t& p, double* a) {
    const double v[kPlanFields] = {(double)p.variant, (double)p.cluster_size, (double)p.threads,
                                   (double)p.waves, (double)p.smem_bytes, (double)p.workspace_bytes,
                                   (double)p.slice_elems, (double)p.active_clusters,
                                   (double)p.ctas_per_sm, (double)p.chunk_elems,
                                   (double)p.ring_slots, (double)p.rows_per_cluster,
                                   (double)p.exchange, (double)p.pred_us,
                                   (double)p.pred_two_pass_us, (double)p.staged_elems};
    std::memcpy(a, v, sizeof(v));
}

// Re-derive a stored plan on `dev`: the launch fields come from the planner,
// the choice (variant, cluster size, threads, residency, ring, rows per
// cluster, exchange, staged length) and the predictions from the file.
bool plan_from_array(int dev, const ChosenPlan& key, const std::vector<Json>& a,
                     credit_plan_t* out) {
    if (a.size() != kPlanFields) return false;
    for (const Json& j : a)
        if (j.kind != Json::kNum) return false;
    const credit_variant_t v = (credit_variant_t)(int)a[0].num;
    const int P = (int)a[1].num, threads = (int)a[2].num, cps = (int)a[8].num;
    const int64_t chunk = (int64_t)a[9].num, staged = (int64_t)a[15].num;
    const int rpc = (int)a[11].num, xchg = (int)a[12].num;
    const int64_t slice = (int64_t)a[6].num;
    const bool pers = v == CREDIT_CLUSTER_PERSISTENT || v == CREDIT_CLUSTER_PIPELINED;
    if (v != CREDIT_CLUSTER && v != CREDIT_TWO_PASS && v != CREDIT_WARP_ROWS && !pers) return false;
    if (make_plan(dev, (credit_op_t)key.op, key.rows, key.cols, (credit_dtype_t)key.dtype, v, P,
                  v == CREDIT_CLUSTER || pers ? threads : 0, pers ? cps : 0, out,
                  pers ? chunk : 0, v == CREDIT_CLUSTER ? rpc : 0,
                  v == CREDIT_CLUSTER && staged < slice ? staged : 0) != CREDIT_OK)
        return false;
    if (xchg == CREDIT_EXCHANGE_BARRIER || xchg == CREDIT_EXCHANGE_ASYNC) {
        if (v == CREDIT_CLUSTER || (v == CREDIT_CLUSTER_PERSISTENT))
            out->exchange = xchg;
    }
    out->pred_us = (float)a[13].num;
    out->pred_two_pass_us = (float)a[14].num;
    return true;
}

std::mutex g_env_mu;
bool g_env_loaded[kMaxDevices];

}  // namespace

void profile_env_load(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return;
    const char* path = std::getenv("CREDIT_PROFILE");
    if (!path || !*path) return;
    {
        std::lock_guard<std::mutex> lk(g_env_mu);
        if (g_env_loaded[dev]) return;
        g_env_loaded[dev] = true;
    }
    credit_load_profile(dev, path);  // a missing or stale file just means no head start
}

void profile_env_save(int dev) {
    const char* path = std::getenv("CREDIT_PROFILE");
    if (path && *path) credit_save_profile(dev, path);
}

bool forced_plan(int dev, credit_op_t op, int64_t rows, int64_t cols, credit_dtype_t dtype,
                 credit_plan_t* out) {
    const char* f = std::getenv("CREDIT_FORCE");
    if (!f || !*f) return false;
    const std::string s(f);
    if (s == "twopass" || s == "two_pass")
        return make_plan(dev, op, rows, cols, dtype, CREDIT_TWO_PASS, 0, 0, 0, out) == CREDIT_OK;
    if (s == "warp_rows")
        return make_plan(dev, op, rows, cols, dtype, CREDIT_WARP_ROWS, 1, 0, 0, out) == CREDIT_OK;
    const size_t c1 = s.find(':');
    if (c1 == std::string::npos) return false;
    const std::string kind = s.substr(0, c1);
    const char* q = s.c_str() + c1 + 1;
    char* e = nullptr;
    const long P = std::strtol(q, &e, 10);
    if (e == q || P < 1 || P > kMaxCluster) return false;
    long R = 0, staged = 0;
    if (*e == 'x') {
        q = e + 1;
        R = std::strtol(q, &e, 10);
        if (e == q) return false;
    }
    if (*e == ':' && e[1] == 's') {
        q = e + 2;
        staged = std::strtol(q, &e, 10);
        if (e == q || staged < 1) return false;
    }
    long threads = 0;
    if (*e == ':' && e[1] == 't') {
        q = e + 2;
        threads = std::strtol(q, &e, 10);
        if (e == q || threads < 32 || threads > 1024 || threads % 32) return false;
    }
    if (*e) return false;
    credit_variant_t v;
    if (kind == "cluster") v = CREDIT_CLUSTER;
    else if (kind == "persist") v = CREDIT_CLUSTER_PERSISTENT;
    else if (kind == "pipe") v = CREDIT_CLUSTER_PIPELINED;
    else return false;
    if (v != CREDIT_CLUSTER && (R || staged || threads)) return false;
    return make_plan(dev, op, rows, cols, dtype, v, (int)P, (int)threads, 0, out, 0, (int)R,
                     staged) == CREDIT_OK;
}

}  // namespace credit

using namespace credit;

extern "C" {

credit_status_t credit_device_key(int device, credit_device_key_t* out) {
    if (!out || device < 0 || device >= kMaxDevices) return CREDIT_ERR_INVALID_ARG;
    return device_key(device, out) ? CREDIT_OK : CREDIT_ERR_CUDA;
}

credit_status_t credit_profile_check(const char* path, const credit_device_key_t* key) {
    if (!path || !key) return CREDIT_ERR_INVALID_ARG;
    std::string text;
    Json root;
    if (!read_file(path, &text) || !parse(text, &root)) return CREDIT_ERR_INVALID_ARG;
    return check(root, *key);
}

credit_status_t credit_save_profile(int device, const char* path) {
    if (!path || device < 0 || device >= kMaxDevices) return CREDIT_ERR_INVALID_ARG;
    credit_device_key_t key;
    if (!device_key(device, &key)) return CREDIT_ERR_CUDA;
    const std::string tmp = std::string(path) + ".tmp";
    FILE* f = std::fopen(tmp.c_str(), "w");
    if (!f) return CREDIT_ERR_INVALID_ARG;
    std::fprintf(f, "{\"format\": \"%s\", \"library\": \"%s\",\n", kFormat, credit_version());
    std::fprintf(f,
                 " \"device\": {\"name\": \"%s\", \"sms\": %d, \"sm_clock_mhz\": %d, "
                 "\"mem_clock_mhz\": %d, \"cc_major\": %d, \"cc_minor\": %d},\n",
                 escaped(key.gpu_name).c_str(), key.sms, key.sm_clock_mhz, key.mem_clock_mhz,
                 key.cc_major, key.cc_minor);
    DsmemData dd;
    if (dsmem_profile_get(device, &dd)) {
        const char* names[3] = {"barrier_ns", "exchange_ns", "async_exchange_ns"};
        const double* arrs[3] = {dd.barrier_ns, dd.exchange_ns, dd.async_ns};
        std::fprintf(f, " \"dsmem\": {");
        for (int k = 0; k < 3; ++k) {
            std::fprintf(f, "%s\"%s\": [", k ? ", " : "", names[k]);
            for (int P = 0; P <= kMaxCluster; ++P)
                std::fprintf(f, "%s%.3f", P ? ", " : "", arrs[k][P]);
            std::fprintf(f, "]");
        }
        std::fprintf(f, ", \"local_load_ns\": %.3f},\n", dd.local_load_ns);
    }
    std::fprintf(f, " \"local_rates\": [");
    const std::vector<LocalRates> lr = local_rates(device);
    for (size_t i = 0; i < lr.size(); ++i) {
        const LocalRates& r = lr[i];
        std::fprintf(f, "%s\n  {\"op\": %d, \"dtype\": %d, \"pdtype\": %d, \"full\": [",
                     i ? "," : "", r.op, r.dtype, r.pdt);
        for (int c = 0; c <= kLocalMaxCps; ++c) std::fprintf(f, "%s%.3f", c ? ", " : "", r.full[c]);
        std::fprintf(f, "], \"tail50\": [");
        for (int c = 0; c <= kLocalMaxCps; ++c) std::fprintf(f, "%s%.3f", c ? ", " : "", r.tail50[c]);
        std::fprintf(f, "], \"tail75\": [");
        for (int c = 0; c <= kLocalMaxCps; ++c) std::fprintf(f, "%s%.3f", c ? ", " : "", r.tail75[c]);
        std::fprintf(f, "], \"sync\": [");
        for (int P = 0; P < kProfileSizes; ++P) std::fprintf(f, "%s%.5f", P ? ", " : "", r.sync[P]);
        std::fprintf(f, "]}");
    }
    std::fprintf(f, "],\n");
    std::fprintf(f, " \"plans\": [");
    const std::vector<ChosenPlan> plans = chosen_plans(device);
    for (size_t i = 0; i < plans.size(); ++i) {
        const ChosenPlan& c = plans[i];
        double a[kPlanFields];
        plan_to_array(c.plan, a);
        std::fprintf(f, "%s\n  {\"op\": %d, \"dtype\": %d, \"rows\": %lld, \"cols\": %lld, \"plan\": [",
                     i ? "," : "", c.op, c.dtype, (long long)c.rows, (long long)c.cols);
        for (int k = 0; k < kPlanFields; ++k) std::fprintf(f, "%s%.9g", k ? ", " : "", a[k]);
        std::fprintf(f, "]}");
    }
    std::fprintf(f, "]}\n");
    const bool ok = std::fflush(f) == 0 && !std::ferror(f);
    std::fclose(f);
    if (!ok || std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return CREDIT_ERR_INVALID_ARG;
    }
    return CREDIT_OK;
}

credit_status_t credit_load_profile(int device, const char* path) {
    if (!path || device < 0 || device >= kMaxDevices) return CREDIT_ERR_INVALID_ARG;
    credit_device_key_t key;
    if (!device_key(device, &key)) return CREDIT_ERR_CUDA;
    std::string text;
    Json root;
    if (!read_file(path, &text) || !parse(text, &root)) return CREDIT_ERR_INVALID_ARG;
    const credit_status_t st = check(root, key);
    if (st != CREDIT_OK) return st;
    if (const Json* d = root.get("dsmem")) {
        const char* names[3] = {"barrier_ns", "exchange_ns", "async_exchange_ns"};
        DsmemData dd;
        double* arrs[3] = {dd.barrier_ns, dd.exchange_ns, dd.async_ns};
        bool good = d->kind == Json::kObj;
        for (int k = 0; good && k < 3; ++k) {
            const Json* a = d->get(names[k]);
            good = a && a->kind == Json::kArr && a->arr.size() == (size_t)kMaxCluster + 1;
            for (int P = 0; good && P <= kMaxCluster; ++P) {
                good = a->arr[P].kind == Json::kNum && a->arr[P].num >= 0.0;
                if (good) arrs[k][P] = a->arr[P].num;
            }
        }
        dd.local_load_ns = num_or(d->get("local_load_ns"), -1.0);
        if (!good || dd.local_load_ns < 0.0) return CREDIT_ERR_INVALID_ARG;
        dsmem_profile_set(device, dd);
    }
    if (const Json* l = root.get("local_rates")) {
        if (l->kind != Json::kArr) return CREDIT_ERR_INVALID_ARG;
        for (const Json& e : l->arr) {
            LocalRates r;
            r.op = (int)num_or(e.get("op"), -1);
            r.dtype = (int)num_or(e.get("dtype"), -1);
            r.pdt = (int)num_or(e.get("pdtype"), -2);
            const Json* arrs[3] = {e.get("full"), e.get("tail50"), e.get("tail75")};
            double* dst[3] = {r.full, r.tail50, r.tail75};
            bool good = r.op >= 0 && r.op <= CREDIT_PEARSON && (r.dtype == 0 || r.dtype == 1) &&
                        r.pdt >= -1 && r.pdt <= 1;
            for (int k = 0; good && k < 3; ++k) {
                good = arrs[k] && arrs[k]->kind == Json::kArr &&
                       arrs[k]->arr.size() == (size_t)kLocalMaxCps + 1;
                for (int c = 0; good && c <= kLocalMaxCps; ++c) {
                    good = arrs[k]->arr[c].kind == Json::kNum && arrs[k]->arr[c].num >= 0.0;
                    if (good) dst[k][c] = arrs[k]->arr[c].num;
                }
            }
            const Json* sy = e.get("sync");
            good = good && sy && sy->kind == Json::kArr && sy->arr.size() == (size_t)kProfileSizes;
            for (int P = 0; good && P < kProfileSizes; ++P) {
                good = sy->arr[P].kind == Json::kNum && sy->arr[P].num >= 0.0;
                if (good) r.sync[P] = sy->arr[P].num;
            }
            if (!good) return CREDIT_ERR_INVALID_ARG;
            local_rates_put(device, r);
        }
    }
    if (const Json* plans = root.get("plans")) {
        if (plans->kind != Json::kArr) return CREDIT_ERR_INVALID_ARG;
        for (const Json& e : plans->arr) {
            const Json* pl = e.get("plan");
            if (!pl || pl->kind != Json::kArr) return CREDIT_ERR_INVALID_ARG;
            ChosenPlan c;
            c.op = (int)num_or(e.get("op"), -1);
            c.dtype = (int)num_or(e.get("dtype"), -1);
            c.rows = (int64_t)num_or(e.get("rows"), 0);
            c.cols = (int64_t)num_or(e.get("cols"), 0);
            if (c.op < 0 || c.op > CREDIT_PEARSON || (c.dtype != CREDIT_F32 && c.dtype != CREDIT_BF16) ||
                c.rows < 1 || c.cols < 1)
                return CREDIT_ERR_INVALID_ARG;
            // a plan this device cannot launch is skipped, not fatal
            if (plan_from_array(device, c, pl->arr, &c.plan)) chosen_plan_put(device, c);
        }
    }
    return CREDIT_OK;
}

}  // extern "C"
