"""A7: the loss-scale bookkeeping of fp16 training, restated for the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring): it shares nothing with
the library's own scaler and imports nothing of the product.

What the pages fix:
  - distrib_optimizer page, "MixedPrecisionOptimizer" layer (the grad_scaler
    argument): fp16 training always needs a grad scaler; with bf16 it may be
    absent, or a constant one.
  - ipipp.com Megatron/DeepSpeed page, the mixed-parallel configuration
    example: fp16 with "loss_scale": 0 (a dynamic scale) and
    "initial_scale_power": 16, so the scale starts at 2^16.
  - distrib_optimizer page, the step skeleton: prepare_grads reports found_inf
    and a step that found an inf/NaN is skipped.

What they leave open, and the reading taken (the usual dynamic loss scaling):
  - an overflow step uses one hysteresis strike; once the strikes are used
    up, the scale is multiplied by the backoff factor (0.5: halved), never
    below min_scale;
  - after growth_interval clean steps in a row the scale is multiplied by
    the growth factor (2) and the hysteresis strikes are restored;
  - an overflow step clears the run of clean steps.
With a hysteresis of 1 this is the backoff/growth rule of torch's GradScaler.
"""

import math


def initial_scale(initial_scale_power=16):
    """The dynamic scale's start value from the DeepSpeed fp16 setting
    initial_scale_power: 2 raised to that power."""
    return math.ldexp(1.0, int(initial_scale_power))


class LossScale:
    """Host state of the dynamic loss scale; update() after every step."""

    def __init__(self, scale=None, growth_factor=2.0, backoff_factor=0.5, growth_interval=1000,
                 hysteresis=1, min_scale=1.0):
        self.scale = initial_scale() if scale is None else float(scale)
        self.growth_factor = float(growth_factor)
        self.backoff_factor = float(backoff_factor)
        self.growth_interval = int(growth_interval)
        self.hysteresis = int(hysteresis)
        self.min_scale = float(min_scale)
        self.clean_steps = 0                  # clean steps in a row since the last change
        self.strikes_left = self.hysteresis  # overflows still absorbed before a backoff

    def update(self, found_inf):
        """Advances the scale past one step that found (or did not find) an
        inf/NaN in its grads.  Returns the scale for the next step."""
        if found_inf:
            self.clean_steps = 0
            self.strikes_left -= 1
            if self.strikes_left <= 0:
                self.scale = max(self.scale * self.backoff_factor, self.min_scale)
        else:
            self.clean_steps += 1
            if self.clean_steps == self.growth_interval:
                self.scale = self.scale * self.growth_factor
                self.clean_steps = 0
                self.strikes_left = self.hysteresis
        return self.scale

    def inv_scale(self):
        """1 / scale rounded once to fp32: the factor that unscales the main
        grads in prepare_grads."""
        import numpy as np
        return float(np.float32(1.0 / self.scale))
