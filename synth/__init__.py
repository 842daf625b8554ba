"""Seeded synthetic inputs for the GPULZ coder (shared by tests, oracle checks and bench).

This module holds no part of the coder's arithmetic: it only produces the
Lorenzo-quantized integer code streams that the coder compresses. See
``synth.fields`` for the recipe.
"""
from .fields import CONFIGS, Config, generate, generate_field, lorenzo_codes  # noqa: F401
