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
