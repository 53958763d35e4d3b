"""CPU oracle for the MLP training step (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  See mlp_oracle.py for what it computes and which passage each
step follows.
"""
from .mlp_oracle import *  # noqa: F401,F403
from .mlp_oracle import (rne_bf16, act_forward, gelu_tanh_grad, linear,  # noqa: F401
                         softmax_ce, argmax_rows, adamw, forward, backward,
                         train_step, run_steps)
