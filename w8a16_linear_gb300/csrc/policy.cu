// Fail-closed parser of a checkpoint's diffusion_step_policy (JSON), host only.
//
// TensorRT-LLM PR #17476, "Load static FP8 Cosmos3 Nano/Super checkpoints
// without re-quantizing them", section Denoising-step activation precision:
// the producer publishes the policy under
// quantization_config.runtime.diffusion_step_policy, and policy shapes that
// are not implemented are refused rather than partially honoured -- unknown
// or missing fields, schema_version other than 1, and any other type,
// index_space, default_mode or overlap value (overlap is validated but not
// acted on).  diffusers PR #14664, "[Cosmos3] Mixed W8A8/W8A16 denoising for
// ModelOpt FP8 checkpoints", section Behavior: "runtime: null" means no
// policy (fully quantized) and the reasoner's precision is stated outright.
//
// Accepted document: JSON null, or one flat object with exactly the keys
//   schema_version  integer 1
//   type            "first_last_n"
//   index_space     "scheduler_step"
//   default_mode    "w8a8"
//   overlap         "w8a16"
//   first_steps     integer >= 0
//   last_steps      integer >= 0
//   reasoner        "a16" | "a8"
// (the pages name the fields, not the spellings of the enumerated values;
// these are this library's reading of them).  Anything else -- other keys or
// values, duplicates, non-integer numbers, nested values, escapes, trailing
// text -- is refused with W8_ERR_POLICY.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/w8lin.h"
#include "internal.h"

namespace {

struct Parser {
  const char* p;
  std::string err;

  void ws() {
    while (*p == ' ' || *p == '\t' || *p == '\n' || *p == '\r') ++p;
  }
  bool lit(const char* s) {
    const size_t n = std::strlen(s);
    if (std::strncmp(p, s, n) != 0) return false;
    p += n;
    return true;
  }
  // A JSON string without escapes (none of the accepted values needs one).
  bool str(std::string* out) {
    if (*p != '"') return fail("expected a string");
    ++p;
    out->clear();
    while (*p && *p != '"') {
      if (*p == '\\') return fail("escapes are not accepted");
      if ((unsigned char)*p < 0x20) return fail("control character in string");
      out->push_back(*p++);
    }
    if (*p != '"') return fail("unterminated string");
    ++p;
    return true;
  }
  // A JSON number that is an integer in [-2^31, 2^31).
  bool integer(int64_t* out) {
    const char* s = p;
    bool neg = false;
    if (*p == '-') {
      neg = true;
      ++p;
    }
    if (!(*p >= '0' && *p <= '9')) return fail("expected an integer");
    if (*p == '0' && p[1] >= '0' && p[1] <= '9') return fail("leading zero");
    int64_t v = 0;
    while (*p >= '0' && *p <= '9') {
      v = v * 10 + (*p - '0');
      if (v > (int64_t)1 << 31) return fail("integer out of range");
      ++p;
    }
    if (*p == '.' || *p == 'e' || *p == 'E') {
      p = s;
      return fail("number is not an integer");
    }
    *out = neg ? -v : v;
    if (*out >= ((int64_t)1 << 31)) return fail("integer out of range");
    return true;
  }
  bool fail(const char* m) {
    if (err.empty()) err = m;
    return false;
  }
};

constexpr int kKeys = 8;
const char* const kKeyNames[kKeys] = {"schema_version", "type",       "index_space", "default_mode",
                                      "overlap",        "first_steps", "last_steps", "reasoner"};

}  // namespace

extern "C" w8_status w8_step_policy_parse(const char* json, w8_step_policy* policy_out,
                                          int32_t* reasoner_mode_out) {
  if (!json || !policy_out || !reasoner_mode_out) {
    w8::set_last_error("w8_step_policy_parse: NULL pointer");
    return W8_ERR_NULL;
  }
  Parser P{json, {}};
  auto refuse = [&](const std::string& why) {
    std::string m = "w8_step_policy_parse: " + why;
    w8::set_last_error(m.c_str());
    return W8_ERR_POLICY;
  };
  P.ws();
  if (P.lit("null")) {
    P.ws();
    if (*P.p) return refuse("trailing text after null");
    policy_out->schema_version = 1;
    policy_out->enabled = 0;
    policy_out->first_steps = 0;
    policy_out->last_steps = 0;
    *reasoner_mode_out = -1;
    w8::set_last_error("");
    return W8_OK;
  }
  if (*P.p != '{') return refuse("policy is not an object");
  ++P.p;
  bool seen[kKeys] = {false};
  int64_t ints[kKeys] = {0};
  std::string strs[kKeys];
  P.ws();
  if (*P.p == '}') return refuse("unknown or missing fields");
  for (;;) {
    P.ws();
    std::string key;
    if (!P.str(&key)) return refuse(P.err);
    int k = -1;
    for (int i = 0; i < kKeys; ++i)
      if (key == kKeyNames[i]) k = i;
    if (k < 0) return refuse("unknown field \"" + key + "\"");
    if (seen[k]) return refuse("duplicate field \"" + key + "\"");
    seen[k] = true;
    P.ws();
    if (*P.p != ':') return refuse("expected ':'");
    ++P.p;
    P.ws();
    const bool is_int = (k == 0 || k == 5 || k == 6);
    if (is_int) {
      if (!P.integer(&ints[k])) return refuse(std::string(kKeyNames[k]) + ": " + P.err);
    } else {
      if (!P.str(&strs[k])) return refuse(std::string(kKeyNames[k]) + ": " + P.err);
    }
    P.ws();
    if (*P.p == ',') {
      ++P.p;
      continue;
    }
    if (*P.p == '}') {
      ++P.p;
      break;
    }
    return refuse("expected ',' or '}'");
  }
  P.ws();
  if (*P.p) return refuse("trailing text after the object");
  for (int i = 0; i < kKeys; ++i)
    if (!seen[i]) return refuse(std::string("missing field \"") + kKeyNames[i] + "\"");
  if (ints[0] != 1) return refuse("schema_version is not 1");
  if (strs[1] != "first_last_n") return refuse("type value refused");
  if (strs[2] != "scheduler_step") return refuse("index_space value refused");
  if (strs[3] != "w8a8") return refuse("default_mode value refused");
  if (strs[4] != "w8a16") return refuse("overlap value refused");
  if (ints[5] < 0 || ints[6] < 0) return refuse("negative step window");
  int32_t reasoner;
  if (strs[7] == "a16") reasoner = W8_MODE_A16;
  else if (strs[7] == "a8") reasoner = W8_MODE_A8;
  else return refuse("reasoner value refused");
  policy_out->schema_version = 1;
  policy_out->enabled = 1;
  policy_out->first_steps = (int32_t)ints[5];
  policy_out->last_steps = (int32_t)ints[6];
  *reasoner_mode_out = reasoner;
  w8::set_last_error("");
  return W8_OK;
}
