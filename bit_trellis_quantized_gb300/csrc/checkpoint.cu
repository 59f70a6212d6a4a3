// Checkpoint loader: safetensors shards of an Escha-W2 export, the escha
// leaf contract, and copies of a projection's leaves into device memory.
//
// safetensors: an 8-byte little-endian header length N, N bytes of JSON
// mapping tensor names to {"dtype", "shape", "data_offsets": [begin, end]}
// (offsets relative to the data that follows the header) plus an optional
// "__metadata__" object, then the data.
//
// Leaf contract (hipfire PR #694, commit reading Escha's test suite; model
// card "EschaLabs/Qwen3.6-35B-A3B-Escha-W2", section "Format notes"):
//  * a coded projection <prefix> has exactly the required leaves
//    <prefix>.escha_code, .escha_rin, .escha_rout; a missing one is an error
//    at load, never a decode into noise;
//  * .escha_s_in, .escha_s_out and .escha_config are optional; the scales
//    ship as all ones (already folded into rin / rout) and are never applied;
//    escha_config is informational;
//  * any other leaf named escha_* (the pages' example: escha_rotation_theta,
//    a Givens rotation variant) is rejected by name;
//  * K comes from the code tensor's own shape: last dimension 16 * K.
// Dense export biases (hipfire PR #694, commit on the dense export's biases):
// <prefix>.bias is optional, but a layer ships its biases together or not at
// all, so a layer whose dense coded projections are only partly biased is a
// corrupt checkpoint.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <set>
#include <string>
#include <vector>

#include "escha.h"
#include "kernels.h"

namespace escha_ckpt_impl {

// ---- a small JSON reader (objects, arrays, strings, numbers, literals) ----
struct Json {
    enum Kind { kNull, kBool, kNum, kStr, kArr, kObj } kind = kNull;
    bool b = false;
    double num = 0;
    long long inum = 0;
    bool is_int = false;
    std::string str;
    std::vector<Json> arr;
    std::vector<std::pair<std::string, Json>> obj;
    const Json* get(const std::string& k) const {
        for (const auto& kv : obj)
            if (kv.first == k) return &kv.second;
        return nullptr;
    }
};

struct Parser {
    const char* p;
    const char* end;
    std::string err;
    int depth = 0;

    void ws() {
        while (p < end && (*p == ' ' || *p == '\t' || *p == '\n' || *p == '\r')) ++p;
    }
    bool fail(const char* m) {
        if (err.empty()) err = m;
        return false;
    }
    bool lit(const char* s) {
        const size_t n = strlen(s);
        if ((size_t)(end - p) < n || memcmp(p, s, n) != 0) return fail("bad literal");
        p += n;
        return true;
    }
    static void put_utf8(std::string& o, unsigned cp) {
        if (cp < 0x80) {
            o += static_cast<char>(cp);
        } else if (cp < 0x800) {
            o += static_cast<char>(0xC0 | (cp >> 6));
            o += static_cast<char>(0x80 | (cp & 0x3F));
        } else if (cp < 0x10000) {
            o += static_cast<char>(0xE0 | (cp >> 12));
            o += static_cast<char>(0x80 | ((cp >> 6) & 0x3F));
            o += static_cast<char>(0x80 | (cp & 0x3F));
        } else {
            o += static_cast<char>(0xF0 | (cp >> 18));
            o += static_cast<char>(0x80 | ((cp >> 12) & 0x3F));
            o += static_cast<char>(0x80 | ((cp >> 6) & 0x3F));
            o += static_cast<char>(0x80 | (cp & 0x3F));
        }
    }
    bool hex4(unsigned& v) {
        if (end - p < 4) return fail("short \\u escape");
        v = 0;
        for (int i = 0; i < 4; ++i) {
            const char c = *p++;
            v <<= 4;
            if (c >= '0' && c <= '9') v |= c - '0';
            else if (c >= 'a' && c <= 'f') v |= c - 'a' + 10;
            else if (c >= 'A' && c <= 'F') v |= c - 'A' + 10;
            else return fail("bad \\u escape");
        }
        return true;
    }
    bool string(std::string& o) {
        if (p >= end || *p != '"') return fail("expected string");
        ++p;
        while (p < end && *p != '"') {
            const unsigned char c = static_cast<unsigned char>(*p++);
            if (c < 0x20) return fail("control character in string");
            if (c != '\\') {
                o += static_cast<char>(c);
                continue;
            }
            if (p >= end) return fail("unterminated escape");
            const char e = *p++;
            switch (e) {
                case '"': o += '"'; break;
                case '\\': o += '\\'; break;
                case '/': o += '/'; break;
                case 'b': o += '\b'; break;
                case 'f': o += '\f'; break;
                case 'n': o += '\n'; break;
                case 'r': o += '\r'; break;
                case 't': o += '\t'; break;
                case 'u': {
                    unsigned cp;
                    if (!hex4(cp)) return false;
                    if (cp >= 0xD800 && cp < 0xDC00) {  // surrogate pair
                        unsigned lo;
                        if (end - p < 2 || p[0] != '\\' || p[1] != 'u') return fail("lone surrogate");
                        p += 2;
                        if (!hex4(lo) || lo < 0xDC00 || lo >= 0xE000) return fail("bad surrogate pair");
                        cp = 0x10000 + ((cp - 0xD800) << 10) + (lo - 0xDC00);
                    }
                    put_utf8(o, cp);
                    break;
                }
                default: return fail("bad escape");
            }
        }
        if (p >= end) return fail("unterminated string");
        ++p;
        return true;
    }
    bool number(Json& j) {
        const char* s = p;
        if (p < end && *p == '-') ++p;
        bool frac = false;
        while (p < end && ((*p >= '0' && *p <= '9') || *p == '.' || *p == 'e' || *p == 'E' || *p == '+' || *p == '-')) {
            if (*p == '.' || *p == 'e' || *p == 'E') frac = true;
            ++p;
        }
        if (p == s) return fail("expected value");
        const std::string t(s, p);
        j.kind = Json::kNum;
        char* e = nullptr;
        j.num = strtod(t.c_str(), &e);
        if (!e || *e) return fail("bad number");
        if (!frac) {
            j.inum = strtoll(t.c_str(), &e, 10);
            j.is_int = e && !*e;
        }
        return true;
    }
    bool value(Json& j) {
        if (++depth > 64) return fail("nesting too deep");
        ws();
        if (p >= end) return fail("unexpected end");
        bool ok = true;
        if (*p == '{') {
            ++p;
            j.kind = Json::kObj;
            ws();
            if (p < end && *p == '}') {
                ++p;
            } else {
                for (;;) {
                    ws();
                    std::string k;
                    if (!string(k)) return false;
                    ws();
                    if (p >= end || *p != ':') return fail("expected ':'");
                    ++p;
                    Json v;
                    if (!value(v)) return false;
                    j.obj.emplace_back(std::move(k), std::move(v));
                    ws();
                    if (p < end && *p == ',') {
                        ++p;
                        continue;
                    }
                    if (p < end && *p == '}') {
                        ++p;
                        break;
                    }
                    return fail("expected ',' or '}'");
                }
            }
        } else if (*p == '[') {
            ++p;
            j.kind = Json::kArr;
            ws();
            if (p < end && *p == ']') {
                ++p;
            } else {
                for (;;) {
                    Json v;
                    if (!value(v)) return false;
                    j.arr.push_back(std::move(v));
                    ws();
                    if (p < end && *p == ',') {
                        ++p;
                        continue;
                    }
                    if (p < end && *p == ']') {
                        ++p;
                        break;
                    }
                    return fail("expected ',' or ']'");
                }
            }
        } else if (*p == '"') {
            j.kind = Json::kStr;
            ok = string(j.str);
        } else if (*p == 't') {
            j.kind = Json::kBool;
            j.b = true;
            ok = lit("true");
        } else if (*p == 'f') {
            j.kind = Json::kBool;
            ok = lit("false");
        } else if (*p == 'n') {
            ok = lit("null");
        } else {
            ok = number(j);
        }
        --depth;
        return ok;
    }
};

// ---- tensors and shards ----------------------------------------------------
struct Tensor {
    std::string name, dtype;
    std::vector<long long> shape;
    int shard = 0;
    unsigned long long begin = 0, end = 0;  // absolute byte offsets in the shard file
};

struct Shard {
    std::string path;
};

struct Proj {
    escha_proj_info info{};
    std::string prefix;
    const Tensor* code = nullptr;
    const Tensor* rin = nullptr;
    const Tensor* rout = nullptr;
    const Tensor* bias = nullptr;
};

int dtype_size(const std::string& d) {
    if (d == "F64" || d == "I64" || d == "U64") return 8;
    if (d == "F32" || d == "I32" || d == "U32") return 4;
    if (d == "F16" || d == "BF16" || d == "I16" || d == "U16") return 2;
    if (d == "I8" || d == "U8" || d == "BOOL" || d == "F8_E4M3" || d == "F8_E5M2") return 1;
    return 0;
}

}  // namespace escha_ckpt_impl

struct escha_ckpt {
    std::vector<escha_ckpt_impl::Shard> shards;
    std::map<std::string, escha_ckpt_impl::Tensor> tensors;
    std::vector<escha_ckpt_impl::Proj> projs;
};

namespace {

using escha_ckpt_impl::Json;
using escha_ckpt_impl::Proj;
using escha_ckpt_impl::Tensor;


int ck_fail(int code, const std::string& m) {

    escha::set_last_error(m.c_str());
    return code;
}

struct FileCloser {
    void operator()(FILE* f) const {
        if (f) fclose(f);
    }
};
using File = std::unique_ptr<FILE, FileCloser>;

// Parses one shard's header into c->tensors.
int parse_shard(escha_ckpt* c, int si) {
    const std::string& path = c->shards[si].path;
    File f(fopen(path.c_str(), "rb"));
    if (!f) return ck_fail(ESCHA_E_IO, "checkpoint: cannot open " + path);
    if (fseek(f.get(), 0, SEEK_END) != 0) return ck_fail(ESCHA_E_IO, "checkpoint: cannot seek " + path);
    const long long fsize = ftell(f.get());
    fseek(f.get(), 0, SEEK_SET);
    unsigned char lenb[8];
    if (fsize < 8 || fread(lenb, 1, 8, f.get()) != 8) return ck_fail(ESCHA_E_IO, "checkpoint: " + path + " is too short");
    unsigned long long hlen = 0;
    for (int i = 7; i >= 0; --i) hlen = (hlen << 8) | lenb[i];
    if (hlen == 0 || hlen > (100ull << 20) || (long long)(8 + hlen) > fsize)
        return ck_fail(ESCHA_E_IO, "checkpoint: " + path + " has an invalid header length");
    std::string hdr(hlen, '\0');
    if (fread(&hdr[0], 1, hlen, f.get()) != hlen) return ck_fail(ESCHA_E_IO, "checkpoint: cannot read header of " + path);
    escha_ckpt_impl::Parser ps{hdr.data(), hdr.data() + hdr.size(), std::string(), 0};
    Json root;
    if (!ps.value(root)) return ck_fail(ESCHA_E_IO, "checkpoint: header of " + path + " is not JSON (" + ps.err + ")");
    ps.ws();
    if (ps.p != ps.end || root.kind != Json::kObj)
        return ck_fail(ESCHA_E_IO, "checkpoint: header of " + path + " is not a JSON object");
    const unsigned long long data0 = 8 + hlen, dsize = (unsigned long long)fsize - data0;
    for (const auto& kv : root.obj) {
        if (kv.first == "__metadata__") continue;
        const Json& t = kv.second;
        const Json* dt = t.get("dtype");
        const Json* sh = t.get("shape");
        const Json* off = t.get("data_offsets");
        if (t.kind != Json::kObj || !dt || dt->kind != Json::kStr || !sh || sh->kind != Json::kArr || !off ||
            off->kind != Json::kArr || off->arr.size() != 2)
            return ck_fail(ESCHA_E_IO, "checkpoint: malformed entry for tensor " + kv.first + " in " + path);
        Tensor x;
        x.name = kv.first;
        x.dtype = dt->str;
        x.shard = si;
        const int es = escha_ckpt_impl::dtype_size(x.dtype);
        if (!es) return ck_fail(ESCHA_E_IO, "checkpoint: unknown dtype " + x.dtype + " of tensor " + kv.first);
        // element count, checked against the shard's data size before every
        // multiply, so a claimed shape cannot wrap around 64 bits
        const unsigned long long max_n = dsize / static_cast<unsigned long long>(es);
        unsigned long long n = 1;
        bool empty = false;
        for (const Json& d : sh->arr) {
            if (d.kind != Json::kNum || !d.is_int || d.inum < 0 || d.inum > (1ll << 40))
                return ck_fail(ESCHA_E_IO, "checkpoint: bad shape of tensor " + kv.first);
            x.shape.push_back(d.inum);
            const unsigned long long dim = static_cast<unsigned long long>(d.inum);
            if (dim == 0) empty = true;
            if (!empty && dim > 0 && n > max_n / dim)
                return ck_fail(ESCHA_E_IO, "checkpoint: shape of tensor " + kv.first + " exceeds its shard's data");
            n = empty ? 0 : n * dim;
        }
        for (const Json& o : off->arr)
            if (o.kind != Json::kNum || !o.is_int || o.inum < 0)
                return ck_fail(ESCHA_E_IO, "checkpoint: bad data_offsets of tensor " + kv.first);
        const unsigned long long b = off->arr[0].inum, e = off->arr[1].inum;
        if (e < b || e > dsize || e - b != n * es)
            return ck_fail(ESCHA_E_IO, "checkpoint: data_offsets of tensor " + kv.first + " do not match its shape");
        x.begin = data0 + b;
        x.end = data0 + e;
        if (c->tensors.count(x.name)) return ck_fail(ESCHA_E_CKPT, "checkpoint: tensor " + x.name + " appears twice");
        c->tensors.emplace(x.name, std::move(x));
    }
    return ESCHA_OK;
}

// "model.layers.12.mlp.gate_proj" -> "model.layers.12."; no layer index -> the prefix itself
std::string layer_key(const std::string& prefix) {
    size_t pos = 0;
    while ((pos = prefix.find("layers.", pos)) != std::string::npos) {
        size_t q = pos + 7;
        size_t r = q;
        while (r < prefix.size() && prefix[r] >= '0' && prefix[r] <= '9') ++r;
        if (r > q && r < prefix.size() && prefix[r] == '.') return prefix.substr(0, r + 1);
        pos = q;
    }
    return prefix;
}

bool all_ones(const escha_ckpt* c, const Tensor& t) {
    const size_t n = t.end - t.begin;
    std::vector<unsigned char> buf(n);
    File f(fopen(c->shards[t.shard].path.c_str(), "rb"));
    if (!f || fseek(f.get(), static_cast<long>(t.begin), SEEK_SET) != 0 || fread(buf.data(), 1, n, f.get()) != n)
        return false;
    if (t.dtype == "F16") {
        for (size_t i = 0; i + 1 < n; i += 2)
            if (buf[i] != 0x00 || buf[i + 1] != 0x3C) return false;  // 1.0 = 0x3C00
        return true;
    }
    if (t.dtype == "F32") {
        for (size_t i = 0; i + 3 < n; i += 4)
            if (buf[i] || buf[i + 1] || buf[i + 2] != 0x80 || buf[i + 3] != 0x3F) return false;  // 0x3F800000
        return true;
    }
    if (t.dtype == "BF16") {
        for (size_t i = 0; i + 1 < n; i += 2)
            if (buf[i] != 0x80 || buf[i + 1] != 0x3F) return false;  // 0x3F80
        return true;
    }
    return false;
}

int validate(escha_ckpt* c) {
    static const std::set<std::string> kKnown = {"escha_code", "escha_rin", "escha_rout",
                                                 "escha_s_in", "escha_s_out", "escha_config"};
    std::map<std::string, std::map<std::string, const Tensor*>> groups;  // prefix -> leaf -> tensor
    for (const auto& kv : c->tensors) {
        const std::string& name = kv.first;
        const size_t dot = name.rfind('.');
        const std::string leaf = dot == std::string::npos ? name : name.substr(dot + 1);
        if (leaf.compare(0, 6, "escha_") != 0) continue;
        if (!kKnown.count(leaf))
            return ck_fail(ESCHA_E_CKPT, "checkpoint: unsupported escha leaf '" + leaf + "' (tensor " + name +
                                             "); only escha_code/rin/rout/s_in/s_out/config are defined");
        if (dot == std::string::npos) return ck_fail(ESCHA_E_CKPT, "checkpoint: escha leaf without a prefix: " + name);
        groups[name.substr(0, dot)][leaf] = &kv.second;
    }
    for (const auto& g : groups) {
        const std::string& prefix = g.first;
        const auto& L = g.second;
        for (const char* req : {"escha_code", "escha_rin", "escha_rout"})
            if (!L.count(req))
                return ck_fail(ESCHA_E_CKPT, "checkpoint: projection " + prefix + " lacks the required leaf " + req);
        Proj pj;
        pj.prefix = prefix;
        pj.code = L.at("escha_code");
        pj.rin = L.at("escha_rin");
        pj.rout = L.at("escha_rout");
        const Tensor& code = *pj.code;
        if (code.dtype != "I16" && code.dtype != "U16")
            return ck_fail(ESCHA_E_CKPT, "checkpoint: " + code.name + " has dtype " + code.dtype + ", not I16/U16");
        if (code.shape.size() != 3 && code.shape.size() != 4)
            return ck_fail(ESCHA_E_CKPT, "checkpoint: " + code.name + " must be [in/16][out/16][16K] or [E][in/16][out/16][16K]");
        const long long last = code.shape.back();
        if (last != 32 && last != 48)
            return ck_fail(ESCHA_E_CKPT, "checkpoint: " + code.name + " last dimension " + std::to_string(last) +
                                             " is not 16*K with K in {2, 3}");
        const bool experts = code.shape.size() == 4;
        const long long E = experts ? code.shape[0] : 0;
        const long long in = 16 * code.shape[code.shape.size() - 3], out = 16 * code.shape[code.shape.size() - 2];
        if (in <= 0 || out <= 0 || in > (1 << 30) || out > (1 << 30) || (experts && E <= 0))
            return ck_fail(ESCHA_E_CKPT, "checkpoint: " + code.name + " has an empty or oversized grid");
        auto vec_ok = [&](const Tensor* t, long long n) {
            if (t->dtype != "F16") return false;
            if (experts) return t->shape.size() == 2 && t->shape[0] == E && t->shape[1] == n;
            return t->shape.size() == 1 && t->shape[0] == n;
        };
        if (!vec_ok(pj.rin, in))
            return ck_fail(ESCHA_E_CKPT, "checkpoint: " + pj.rin->name + " must be F16 [" + (experts ? "E][" : "") +
                                             std::to_string(in) + "]");
        if (!vec_ok(pj.rout, out))
            return ck_fail(ESCHA_E_CKPT, "checkpoint: " + pj.rout->name + " must be F16 [" + (experts ? "E][" : "") +
                                             std::to_string(out) + "]");
        escha_proj_info& I = pj.info;
        snprintf(I.prefix, sizeof(I.prefix), "%s", prefix.c_str());
        if (prefix.size() >= sizeof(I.prefix))
            return ck_fail(ESCHA_E_CKPT, "checkpoint: projection name longer than 255 bytes: " + prefix);
        I.K = static_cast<int>(last / 16);
        I.n_experts = static_cast<int>(E);
        I.in = static_cast<int>(in);
        I.out = static_cast<int>(out);
        I.has_s_in = L.count("escha_s_in") ? 1 : 0;
        I.has_s_out = L.count("escha_s_out") ? 1 : 0;
        I.has_config = L.count("escha_config") ? 1 : 0;
        I.scales_all_ones = 1;
        for (const char* s : {"escha_s_in", "escha_s_out"})
            if (L.count(s) && !all_ones(c, *L.at(s))) I.scales_all_ones = 0;
        I.config_k = -1;
        if (I.has_config) {
            const Tensor& cf = *L.at("escha_config");
            if (cf.dtype == "I32" && !cf.shape.empty() && cf.shape.back() == 9 && cf.end - cf.begin >= 8) {
                int32_t v[2] = {0, 0};
                File f(fopen(c->shards[cf.shard].path.c_str(), "rb"));
                if (f && fseek(f.get(), static_cast<long>(cf.begin), SEEK_SET) == 0 && fread(v, 4, 2, f.get()) == 2)
                    I.config_k = v[1];
            }
        }
        auto bt = c->tensors.find(prefix + ".bias");
        if (bt != c->tensors.end()) {
            const Tensor& b = bt->second;
            const bool ok_t = b.dtype == "F32" || b.dtype == "F16" || b.dtype == "BF16";
            if (experts || !ok_t || b.shape.size() != 1 || b.shape[0] != out)
                return ck_fail(ESCHA_E_CKPT, "checkpoint: " + b.name + " must be an F32/F16/BF16 vector of " +
                                                 std::to_string(out) + " on a dense projection");
            pj.bias = &b;
            I.has_bias = 1;
        }
        c->projs.push_back(pj);
    }
    // a layer's dense coded projections carry biases together or not at all
    std::map<std::string, std::pair<int, int>> per_layer;  // key -> (dense projections, biased)
    for (const Proj& pj : c->projs) {
        if (pj.info.n_experts) continue;
        auto& v = per_layer[layer_key(pj.prefix)];
        ++v.first;
        v.second += pj.info.has_bias;
    }
    for (const auto& kv : per_layer)
        if (kv.second.second != 0 && kv.second.second != kv.second.first)
            return ck_fail(ESCHA_E_CKPT, "checkpoint: layer " + kv.first + " biases only " +
                                             std::to_string(kv.second.second) + " of its " +
                                             std::to_string(kv.second.first) + " coded projections");
    return ESCHA_OK;
}

// Reads a tensor's bytes into host memory.
int read_host(const escha_ckpt* c, const Tensor& t, void* dst) {
    File f(fopen(c->shards[t.shard].path.c_str(), "rb"));
    const size_t n = t.end - t.begin;
    if (!f || fseek(f.get(), static_cast<long>(t.begin), SEEK_SET) != 0 || fread(dst, 1, n, f.get()) != n)
        return ck_fail(ESCHA_E_IO, "checkpoint: cannot read tensor " + t.name);
    return ESCHA_OK;
}

int copy_to_device(const escha_ckpt* c, const Tensor& t, void* dst, cudaStream_t s) {
    std::vector<unsigned char> buf(t.end - t.begin);
    int r = read_host(c, t, buf.data());
    if (r) return r;
    cudaError_t e = cudaMemcpyAsync(dst, buf.data(), buf.size(), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the staging buffer goes out of scope
    if (e != cudaSuccess) return ck_fail(ESCHA_E_CUDA, std::string("checkpoint: copy failed: ") + cudaGetErrorString(e));
    return ESCHA_OK;
}

float half_bits_to_float(uint16_t h, bool bf16) {
    if (bf16) {
        const uint32_t u = static_cast<uint32_t>(h) << 16;
        float f;
        memcpy(&f, &u, 4);
        return f;
    }
    const uint32_t sign = (h & 0x8000u) << 16, exp = (h >> 10) & 0x1F, man = h & 0x3FF;
    uint32_t u;
    if (exp == 0x1F) {
        u = sign | 0x7F800000u | (man << 13);
    } else if (exp == 0) {
        if (man == 0) {
            u = sign;
        } else {  // subnormal: renormalise
            int e = -1;
            uint32_t m = man;
            do {
                m <<= 1;
                ++e;
            } while (!(m & 0x400));
            u = sign | (static_cast<uint32_t>(127 - 15 - e) << 23) | ((m & 0x3FF) << 13);
        }
    } else {
        u = sign | ((exp + 112) << 23) | (man << 13);
    }
    float f;
    memcpy(&f, &u, 4);
    return f;
}

}  // namespace

extern "C" {

int escha_ckpt_open(const char* const* paths, int n_paths, escha_ckpt** out) {
    if (!out) return ck_fail(ESCHA_E_ARG, "ckpt_open: out is null");
    *out = nullptr;
    if (!paths || n_paths < 1) return ck_fail(ESCHA_E_ARG, "ckpt_open: no shard paths");
    std::unique_ptr<escha_ckpt> c(new escha_ckpt);
    for (int i = 0; i < n_paths; ++i) {
        if (!paths[i]) return ck_fail(ESCHA_E_ARG, "ckpt_open: a shard path is null");
        c->shards.push_back({paths[i]});
    }
    for (int i = 0; i < n_paths; ++i) {
        const int r = parse_shard(c.get(), i);
        if (r) return r;
    }
    const int r = validate(c.get());
    if (r) return r;
    *out = c.release();
    return ESCHA_OK;
}

void escha_ckpt_close(escha_ckpt* c) { delete c; }

int escha_ckpt_num_projections(const escha_ckpt* c) { return c ? static_cast<int>(c->projs.size()) : 0; }

int escha_ckpt_projection(const escha_ckpt* c, int i, escha_proj_info* info) {
    if (!c || !info) return ck_fail(ESCHA_E_ARG, "ckpt_projection: null argument");
    if (i < 0 || i >= static_cast<int>(c->projs.size()))
        return ck_fail(ESCHA_E_ARG, "ckpt_projection: index " + std::to_string(i) + " out of range");
    *info = c->projs[i].info;
    return ESCHA_OK;
}

int escha_ckpt_tensor_info(const escha_ckpt* c, const char* name, escha_tensor_info* info) {
    if (!c || !name || !info) return ck_fail(ESCHA_E_ARG, "ckpt_tensor_info: null argument");
    auto it = c->tensors.find(name);
    if (it == c->tensors.end()) return ck_fail(ESCHA_E_ARG, std::string("ckpt_tensor_info: no tensor ") + name);
    const Tensor& t = it->second;
    if (t.shape.size() > 8) return ck_fail(ESCHA_E_ARG, "ckpt_tensor_info: rank above 8");
    memset(info, 0, sizeof(*info));
    snprintf(info->dtype, sizeof(info->dtype), "%s", t.dtype.c_str());
    info->ndim = static_cast<int>(t.shape.size());
    for (size_t d = 0; d < t.shape.size(); ++d) info->shape[d] = t.shape[d];
    info->nbytes = t.end - t.begin;
    return ESCHA_OK;
}

int escha_ckpt_read(const escha_ckpt* c, const char* name, void* dst, size_t dst_bytes, int dst_device, void* stream) {
    if (!c || !name || !dst) return ck_fail(ESCHA_E_ARG, "ckpt_read: null argument");
    auto it = c->tensors.find(name);
    if (it == c->tensors.end()) return ck_fail(ESCHA_E_ARG, std::string("ckpt_read: no tensor ") + name);
    const Tensor& t = it->second;
    if (dst_bytes < t.end - t.begin) return ck_fail(ESCHA_E_ARG, std::string("ckpt_read: buffer too small for ") + name);
    if (!dst_device) return read_host(c, t, dst);
    return copy_to_device(c, t, dst, static_cast<cudaStream_t>(stream));
}

int escha_ckpt_load_projection(const escha_ckpt* c, int i, uint16_t* codes, uint16_t* rin, uint16_t* rout,
                               float* bias, int nt_major, void* stream) {
    if (!c || !codes || !rin || !rout) return ck_fail(ESCHA_E_ARG, "ckpt_load_projection: null argument");
    if (i < 0 || i >= static_cast<int>(c->projs.size()))
        return ck_fail(ESCHA_E_ARG, "ckpt_load_projection: index " + std::to_string(i) + " out of range");
    const Proj& pj = c->projs[i];
    if (nt_major != 0 && nt_major != 1) return ck_fail(ESCHA_E_ARG, "ckpt_load_projection: nt_major must be 0 or 1");
    if (nt_major && pj.info.n_experts)
        return ck_fail(ESCHA_E_ARG, "ckpt_load_projection: expert code tensors stay kt-major");
    if (bias && !pj.bias) return ck_fail(ESCHA_E_ARG, "ckpt_load_projection: " + pj.prefix + " has no bias");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int r;
    if (!nt_major) {
        if ((r = copy_to_device(c, *pj.code, codes, s))) return r;
    } else {  // whole tiles moved to the nt-major grid in host memory, then one copy (no device scratch)
        const Tensor& t = *pj.code;
        std::vector<unsigned char> src(t.end - t.begin), dst(t.end - t.begin);
        if ((r = read_host(c, t, src.data()))) return r;
        const size_t KT = pj.info.in / 16, NT = pj.info.out / 16, tile = 16 * 2 * static_cast<size_t>(pj.info.K);
        for (size_t kt = 0; kt < KT; ++kt)
            for (size_t nt = 0; nt < NT; ++nt)
                memcpy(dst.data() + (nt * KT + kt) * tile, src.data() + (kt * NT + nt) * tile, tile);
        cudaError_t e = cudaMemcpyAsync(codes, dst.data(), dst.size(), cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the staging buffer goes out of scope
        if (e != cudaSuccess) return ck_fail(ESCHA_E_CUDA, std::string("ckpt_load_projection: ") + cudaGetErrorString(e));
    }
    if ((r = copy_to_device(c, *pj.rin, rin, s))) return r;
    if ((r = copy_to_device(c, *pj.rout, rout, s))) return r;
    if (bias && pj.bias) {  // widened to f32 on the host
        const Tensor& b = *pj.bias;
        std::vector<float> f(static_cast<size_t>(pj.info.out));
        if (b.dtype == "F32") {
            if ((r = read_host(c, b, f.data()))) return r;
        } else {
            std::vector<uint16_t> h(f.size());
            if ((r = read_host(c, b, h.data()))) return r;
            for (size_t k = 0; k < f.size(); ++k) f[k] = half_bits_to_float(h[k], b.dtype == "BF16");
        }
        cudaError_t e = cudaMemcpyAsync(bias, f.data(), f.size() * 4, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return ck_fail(ESCHA_E_CUDA, std::string("ckpt_load_projection: ") + cudaGetErrorString(e));
    }
    return ESCHA_OK;
}

}  // extern "C"
