"""Per-denoising-step precision policy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P3] *Behavior*: the first 3 and last 3 scheduler steps run W8A16, the
middle steps W8A8; precision is chosen once per scheduler step, so the CFG
conditional and unconditional branches agree.  [P3] *Tests*: "1-step stays
native"; 8 steps trace W8A16x3 / W8A8x2 / W8A16x3 and 35 steps
W8A16x3 / W8A8x29 / W8A16x3.  [P4] *Denoising-step activation precision*:
a checkpoint without a policy runs fully quantized; policy shapes that are
not implemented are refused (schema_version other than 1, and so on); the
mitigation keeps the one-step warmup carve-out.

Readings: step indices are zero-based ([P1] *Describe the bug*: step 3 of 8
is the first W8A8 step); the one-step carve-out means a one-step schedule
runs W8A8 on its only step.
"""

from dataclasses import dataclass

A8 = "A8"
A16 = "A16"


class PolicyError(ValueError):
    pass


@dataclass(frozen=True)
class StepPolicy:
    schema_version: int = 1
    enabled: bool = True
    first_steps: int = 3
    last_steps: int = 3


def step_mode(policy, step, num_steps):
    """Precision of scheduler step ``step`` of ``num_steps``: "A8" or "A16"."""
    if num_steps < 1 or not (0 <= step < num_steps):
        raise PolicyError(f"step {step} outside [0, {num_steps})")
    if policy is None or not policy.enabled:
        return A8
    if policy.schema_version != 1:
        raise PolicyError(f"schema_version {policy.schema_version} is not 1")
    if policy.first_steps < 0 or policy.last_steps < 0:
        raise PolicyError("negative step window")
    if num_steps == 1:
        return A8
    if step < policy.first_steps or step >= num_steps - policy.last_steps:
        return A16
    return A8


# ---------------------------------------------------------------- JSON schema
#
# [P4] *Denoising-step activation precision*: the producer publishes the
# policy under quantization_config.runtime.diffusion_step_policy; policy
# shapes that are not implemented are refused rather than partially honoured:
# unknown or missing fields, schema_version other than 1, and any other type,
# index_space, default_mode or overlap value; overlap is validated but not
# acted on.  [P3] *Behavior*: a checkpoint with ``runtime: null`` runs fully
# quantized; the reasoner's precision is stated outright (``reasoner: a16``).
#
# The pages name the fields but not the accepted spellings of the enumerated
# values.  Reading: type "first_last_n" (the first-N / last-N policy),
# index_space "scheduler_step", default_mode "w8a8" (the native path of the
# middle steps), overlap "w8a16" (where the windows meet the 16-bit path wins,
# which is what the step predicate yields), reasoner "a16" or "a8".

POLICY_KEYS = ("schema_version", "type", "index_space", "default_mode", "overlap",
               "first_steps", "last_steps", "reasoner")
_ENUMS = {"type": ("first_last_n",), "index_space": ("scheduler_step",),
          "default_mode": ("w8a8",), "overlap": ("w8a16",), "reasoner": ("a16", "a8")}


def parse_policy(text):
    """Parse a diffusion_step_policy JSON text fail-closed.

    Returns ``(StepPolicy, reasoner)`` where reasoner is "A16", "A8" or None
    (no policy: ``null``).  Raises PolicyError on anything else.
    """
    import json

    if "\\" in text:       # no accepted value needs an escape; none is honoured
        raise PolicyError("escapes are not accepted")

    def pairs(kv):
        keys = [k for k, _ in kv]
        if len(keys) != len(set(keys)):
            raise PolicyError("duplicate key")
        return dict(kv)

    try:
        obj = json.loads(text, object_pairs_hook=pairs,
                         parse_float=lambda s: (_ for _ in ()).throw(PolicyError("number is not an integer")),
                         parse_constant=lambda s: (_ for _ in ()).throw(PolicyError("bad constant")))
    except PolicyError:
        raise
    except ValueError as e:
        raise PolicyError(f"not valid JSON: {e}") from None
    if obj is None:
        return StepPolicy(enabled=False), None
    if not isinstance(obj, dict):
        raise PolicyError("policy is not an object")
    if set(obj) != set(POLICY_KEYS):
        raise PolicyError("unknown or missing fields")
    for k in ("schema_version", "first_steps", "last_steps"):
        if type(obj[k]) is not int:
            raise PolicyError(f"{k} is not an integer")
    if obj["schema_version"] != 1:
        raise PolicyError("schema_version is not 1")
    for k, allowed in _ENUMS.items():
        if not isinstance(obj[k], str) or obj[k] not in allowed:
            raise PolicyError(f"{k} value refused")
    if obj["first_steps"] < 0 or obj["last_steps"] < 0:
        raise PolicyError("negative step window")
    if obj["first_steps"] >= 2 ** 31 or obj["last_steps"] >= 2 ** 31:
        raise PolicyError("step window out of range")
    pol = StepPolicy(schema_version=1, enabled=True, first_steps=obj["first_steps"],
                     last_steps=obj["last_steps"])
    return pol, obj["reasoner"].upper()
